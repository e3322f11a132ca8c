// attend_bwd_tc.cu -- fast backward for bf16 values with d_V = 64 and d_K <= 4.
//
// Same definitions as attend_bwd.cu (gradients through the Cauchy weights of
// "ZETA: Leveraging Z-order Curves for Efficient Top-k Attention", selection
// held fixed), organised like the fast forward:
//
// Query side, one CTA per 64 queries of a chunk:
//   window part  - a pipeline of units (one query's pass over up to 64 selected
//                  keys): the unit's value rows are copied into a two-slot
//                  shared-memory ring by cp.async one unit ahead, g_ij =
//                  dO_i . v_j runs on the tensor cores (the rows as A fragments,
//                  dO_i in column 0 of B), and a lane's two slots accumulate the
//                  pair terms packed: sum w, sum w g, sum g e, sum e,
//                  sum g c (q-k), sum c (q-k) (Cauchy: the same sums on u = w^2
//                  with the constants applied at the end).
//   own chunk    - G = dO . V^T on tensor cores (mma.sync, dO fragments held
//                  in registers, V tiles cp.async-staged), then the same terms
//                  per element.
//   result       - s_i, gbar_i = G / s, dq_i, the query's dgamma share, and a
//                  32-byte record {q_i, 1/s_i, gbar_i} for the key side.
// Key side, one CTA per 64 keys of a chunk:
//   window part  - the queries that selected key j (a transpose of idx sorted
//                  by key, or by 8-key group): a warp walks the lists of its 16
//                  keys as one run, 32 entries per step, the step's dO rows
//                  staged in a ring one step ahead; G = dO_rows . V_keys^T and
//                  dV_keys += dO^T A on the tensor cores, and dk_j += dL/dw_ij
//                  (-2 dw/d(d^2)) (q_i - k_j) summed per key on the tensor
//                  cores as well (one-hot keys times the entries' terms).
//   own chunk    - S^T = V . dO^T on tensor cores, the element-wise terms, then
//                  dV += P^T . dO with P^T re-packed from the accumulator
//                  fragments (their layout is the A-fragment layout).  Where
//                  it applies (C a multiple of 128, H <= 64, aligned inputs)
//                  the separate tcgen05 kernel of bwd_own_tc05.cu does this
//                  part and the walk adds its sums.
// Other weight kernels (flags; reply A3 "Justification for Euclidean Distance
// Claim") swap in their w, dw/d(d^2) and dw/dgamma.  The softmax keeps a running
// shift m per query on the query side (the sums are moved onto a lower shift
// when it appears, exactly: sum g e and sum e also pick up the shift change),
// and records the final m with 1/s and gbar for the key side.
#include <type_traits>

#include "bwd_rec.cuh"
#include "mma.cuh"

namespace zeta {
namespace {

constexpr int T64 = 64;           // rows per CTA tile (queries or keys)
constexpr int DV = 64;
constexpr int THREADS = 128;

// Sums over the warp of 16 values per lane with 16 shuffles (recursive
// halving); lane L returns the total of value (L >> 1).
__device__ __forceinline__ float warp_transpose_sum16(float (&v)[16], int lane) {
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        const float r = __shfl_xor_sync(kFull, b4 ? v[m] : v[m + 8], 16);
        v[m] = (b4 ? v[m + 8] : v[m]) + r;
    }
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const float r = __shfl_xor_sync(kFull, b3 ? v[m] : v[m + 4], 8);
        v[m] = (b3 ? v[m + 4] : v[m]) + r;
    }
#pragma unroll
    for (int m = 0; m < 2; ++m) {
        const float r = __shfl_xor_sync(kFull, b2 ? v[m] : v[m + 2], 4);
        v[m] = (b2 ? v[m + 2] : v[m]) + r;
    }
    {
        const float r = __shfl_xor_sync(kFull, b1 ? v[0] : v[1], 2);
        v[0] = (b1 ? v[1] : v[0]) + r;
    }
    return v[0] + __shfl_xor_sync(kFull, v[0], 1);
}

template <int DK>
__device__ __forceinline__ float dist2k(const float (&a)[4], float4 b) {
    float d = 0.f;
    const float bb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int x = 0; x < DK; ++x) {
        const float e = a[x] - bb[x];
        d = __fmaf_rn(e, e, d);
    }
    return d;
}

// 64 rows x 64 bf16 of a [.., 64] row-major array into a swizzled tile;
// rows at or beyond `end` are zero-filled.
__device__ __forceinline__ void stage_rows(__nv_bfloat16 *tile, const __nv_bfloat16 *base,
                                           int row0, int end) {
#pragma unroll
    for (int r = 0; r < (T64 * DV / 8) / THREADS; ++r) {
        const int id = r * THREADS + threadIdx.x;
        const int row = id >> 3, ch = id & 7;
        const int gr = row0 + row;
        const bool ok = gr < end;
        cp_async16(smem_u32(tile + swz(row, ch)), base + (int64_t)(ok ? gr : row0) * DV + ch * 8,
                   ok ? 16 : 0);
    }
}

// ============================================================ query side ===

// Tiles of the own-chunk part.
struct __align__(16) QOwn {
    __nv_bfloat16 dO[T64 * DV];
    __nv_bfloat16 v[2][T64 * DV];
    float4 kt[2][T64];
};
// Dynamic shared memory of the query side: the window walk's rings (four warps
// x two slots of q_ring_rows(k) value rows), which become the own-chunk tiles
// once every warp's walk is done, then the window part's sums per query and
// (softmax) its shift per query.
__host__ __device__ inline int q_ring_rows(int k) { return k >= 64 ? 64 : (k + 15) & ~15; }
__host__ __device__ inline size_t q_big_bytes(int k) {
    const size_t ring = (size_t)(THREADS / 32) * 2 * q_ring_rows(k) * DV * 2;
    return ring > sizeof(QOwn) ? ring : sizeof(QOwn);
}
__host__ __device__ inline size_t q_smem_bytes(int k) {
    return q_big_bytes(k) + sizeof(float) * T64 * 12 + sizeof(float) * T64;
}

// Accumulators of one query row: x[0] = sum w, x[1] = sum w g, x[2] = sum g e,
// x[3] = sum e, x[4..7] = sum g c (q-k), x[8..11] = sum c (q-k).  Cauchy:
// c = -2 u / gamma^2 and e = 2 (w - u) / gamma with u = w^2, so the sums are
// kept without the constants: x[2] = sum u g, x[3] = sum u, x[4+d] =
// sum u g (q-k)_d, x[8+d] = sum u (q-k)_d (the epilogue applies them).
// With the softmax, e = 2 w (d2 - m) / gamma^3 depends on the shift m: moving
// the sums from shift m to m' = m + dm multiplies every term by
// sc = exp(dm / gamma^2) and subtracts dm 2/gamma^3 w from each e.
struct QAcc {
    float x[12];
    __device__ void rebase(float dm, float sc, float k2) {
        x[2] -= dm * k2 * x[1];
        x[3] -= dm * k2 * x[0];
#pragma unroll
        for (int y = 0; y < 12; ++y) x[y] *= sc;
    }
};

// The same twelve sums for two rows (a, b) at once, packed f32x2; a weight of
// 0 (masked pair) contributes nothing.
struct QAcc2 {
    float2 x[12];
    __device__ void zero() {
#pragma unroll
        for (int y = 0; y < 12; ++y) x[y] = make_float2(0.f, 0.f);
    }
    __device__ void rebase(float2 dm, float2 sc, float2 k2) {
        x[2] = sub2(x[2], mul2(mul2(dm, k2), x[1]));
        x[3] = sub2(x[3], mul2(mul2(dm, k2), x[0]));
#pragma unroll
        for (int y = 0; y < 12; ++y) x[y] = mul2(x[y], sc);
    }
    // m2ig2 = -2/gamma^2, two_ig = 2/gamma, k2 = 2/gamma^3; d2, m only for the softmax.
    template <int DK, int WK>
    __device__ void add(float2 w, float2 d2, float2 m, float2 g, const float2 (&dq)[4],
                        float2 m2ig2, float2 two_ig, float2 k2) {
        if constexpr (WK == kWCauchy) {        // the constant-free sums (see QAcc)
            const float2 u = mul2(w, w), ug = mul2(u, g);
            x[0] = add2(x[0], w);
            x[1] = fma2(w, g, x[1]);
            x[2] = add2(x[2], ug);
            x[3] = add2(x[3], u);
#pragma unroll
            for (int d = 0; d < DK; ++d) {
                x[4 + d] = fma2(ug, dq[d], x[4 + d]);
                x[8 + d] = fma2(u, dq[d], x[8 + d]);
            }
            return;
        }
        float2 c, e;
        if constexpr (WK == kWSoftmax) {
            c = mul2(w, m2ig2);                                   // -2 w / gamma^2
            e = mul2(mul2(w, sub2(d2, m)), k2);                   // 2 w (d2 - m) / gamma^3
        } else if constexpr (WK == kWInvEuclid) {
            c = mul2(mul2(w, w), mul2(w, dup2(-1.f)));            // -w^3
            e = make_float2(0.f, 0.f);
        } else {
            c = mul2(mul2(w, w), m2ig2);                          // -2 w^2 / gamma^2
            e = mul2(mul2(w, sub2(dup2(1.f), w)), two_ig);        // 2 w (1 - w) / gamma
        }
        x[0] = add2(x[0], w);
        x[1] = fma2(w, g, x[1]);
        x[2] = fma2(g, e, x[2]);
        x[3] = add2(x[3], e);
#pragma unroll
        for (int d = 0; d < DK; ++d) {
            const float2 t = mul2(c, dq[d]);
            x[4 + d] = fma2(g, t, x[4 + d]);
            x[8 + d] = add2(x[8 + d], t);
        }
    }
};

// The softmax carries a shift and its rebasing through both parts; it gets
// more registers (three CTAs per SM) instead of spilling.
template <int DK, int WK>
__global__ void __launch_bounds__(THREADS, WK == kWSoftmax ? 3 : 4)
bwd_query_tc(const float *__restrict__ q, const float *__restrict__ kx,
             const __nv_bfloat16 *__restrict__ v, const float *__restrict__ gamma,
             const int32_t *__restrict__ idx, const __nv_bfloat16 *__restrict__ dout,
             float *__restrict__ dq, QRec *__restrict__ rec, float *__restrict__ dg_part,
             int32_t *status, int N, int H, int k, int C, int tiles_per_chunk) {
    extern __shared__ __align__(16) unsigned char qsm[];
    QOwn &own = *reinterpret_cast<QOwn *>(qsm);
    float(*qpart)[12] = reinterpret_cast<float(*)[12]>(qsm + q_big_bytes(k));
    float *qmpart = reinterpret_cast<float *>(qsm + q_big_bytes(k) + sizeof(float) * T64 * 12);
    const int64_t seg = blockIdx.y;
    const int c = blockIdx.x / tiles_per_chunk;
    const int qt = blockIdx.x % tiles_per_chunk;
    const int cC = c * C, cend = cC + C;
    const int i0 = cC + qt * T64;
    const int iend = min(cend, i0 + T64);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float gm = gamma[seg % H];
    const float inv_g2 = __frcp_rn(gm * gm);
    const float inv_g = __frcp_rn(gm);
    const float *kb = kx + seg * (int64_t)N * DK;
    const float *qb = q + seg * (int64_t)N * DK;
    const __nv_bfloat16 *vb = v + seg * (int64_t)N * DV;
    const __nv_bfloat16 *db = dout + seg * (int64_t)N * DV;
    const int nkt = (iend - 1 - cC) / T64 + 1;

    auto load_ktile = [&](int b, int key0) {
        stage_rows(own.v[b], vb, key0, cend);
        if (threadIdx.x < T64) {
            const int key = key0 + threadIdx.x;
            own.kt[b][threadIdx.x] =
                key < cend ? load_k4(kb + (int64_t)key * DK, DK) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    // ---------------------------------------------------- window part ---
    // A unit is one pass of a query over up to 64 selected keys; lane L owns
    // slots L and L+32 (index, coordinates, the pair's weight terms).  Each
    // unit's value rows are copied into a two-slot ring of swizzled 128-byte
    // rows in shared memory (cp.async) one unit ahead, its indices two units
    // ahead, its key coordinates and dO_i one unit ahead in registers.  The dot
    // products g_ij = dO_i . v_j run on the tensor cores: for 16 selected keys,
    // G = V_J . dO_i is one m16n8k16 mma per 16 dimensions, A the staged rows
    // (ldmatrix) and dO_i in column 0 of B; the owner picks g up from the lane
    // holding column 0.
    const int g4 = lane >> 2, s4 = lane & 3;
    const int wq0 = i0 + warp * 16;
    const int nqw = c > 0 ? max(0, min(16, iend - wq0)) : 0;
    const int npass = (k + 63) >> 6;
    const int nunit = nqw * npass;
    const int rr_ring = q_ring_rows(k);
    const uint32_t slot_bytes = (uint32_t)rr_ring * 128u;
    const uint32_t ring = smem_u32(qsm) + (uint32_t)warp * 2u * slot_bytes;
    auto unit_idx = [&](int u, int (&j)[2]) {            // raw indices of unit u
        j[0] = j[1] = -1;
        if (u < nunit) {
            const int r = u / npass, t0 = (u - r * npass) * 64;
            const int32_t *irow = idx + (seg * N + wq0 + r) * (int64_t)k + t0;
#pragma unroll
            for (int s = 0; s < 2; ++s)
                if (t0 + s * 32 + lane < k) j[s] = __ldg(irow + s * 32 + lane);
        }
    };
    auto validate = [&](int (&j)[2]) {                   // keys outside the prefix -> -1
#pragma unroll
        for (int s = 0; s < 2; ++s)
            if (j[s] != -1 && (unsigned)j[s] >= (unsigned)cC) {
                set_status(status, ZETA_ERR_BOUNDS);
                j[s] = -1;
            }
    };
    auto issue = [&](int u, const int (&j)[2]) {         // value rows of unit u
        const int t0 = (u % npass) * 64;
        const int nrows = min(rr_ring, (min(64, k - t0) + 15) & ~15);
        const uint32_t slot = ring + (uint32_t)(u & 1) * slot_bytes;
        for (int h = 0; 4 * h < nrows; ++h) {
            const int row = 4 * h + (lane >> 3), ch = lane & 7;
            const int jr = __shfl_sync(kFull, row < 32 ? j[0] : j[1], row & 31);
            const bool ok = jr >= 0;
            cp_async16(slot + (uint32_t)swz(row, ch) * 2u, vb + (int64_t)(ok ? jr : 0) * DV + ch * 8,
                       ok ? 16 : 0);
        }
        cp_async_commit();
    };
    auto unit_keys = [&](const int (&j)[2], float4 (&kk)[2]) {
#pragma unroll
        for (int s = 0; s < 2; ++s)
            kk[s] = j[s] >= 0 ? load_k4(kb + (int64_t)j[s] * DK, DK) : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    auto unit_dout = [&](int u) -> uint32_t {            // word `lane` of dO_i of unit u
        if (u >= nunit) return 0u;
        const int i = wq0 + u / npass;
        return reinterpret_cast<const uint32_t *>(db + (int64_t)i * DV)[lane];
    };
    const float k2 = 2.f * inv_g2 * inv_g;
    // rows without a window part
    for (int r = nqw; r < 16; ++r) {
        if (lane < 12) qpart[warp * 16 + r][lane] = 0.f;
        if (lane == 0) qmpart[warp * 16 + r] = INFINITY;
    }
    int jc[2], jn[2], jn2[2];
    unit_idx(0, jc);
    validate(jc);
    if (nunit > 0) issue(0, jc);
    float4 kc[2], kn[2];
    unit_keys(jc, kc);
    uint32_t dwc = unit_dout(0), dwn = 0u;
    auto unit_q = [&](int u, float (&x)[4]) {           // q_i of unit u
#pragma unroll
        for (int d = 0; d < 4; ++d)
            x[d] = (u < nunit && d < DK) ? qb[(int64_t)(wq0 + u / npass) * DK + d] : 0.f;
    };
    float qi[4], qn[4];
    unit_q(0, qi);
    unit_idx(1, jn);
    // the lane's two slots packed (x: slot L, y: slot L+32)
    const float2 ig2w = dup2(inv_g2), m2ig2w = dup2(-2.f * inv_g2), two_igw = dup2(2.f * inv_g);
    const float2 k2w = dup2(k2);
    QAcc2 acc;
    acc.zero();
    float mrun = INFINITY;                       // softmax shift of this query
    for (int u = 0; u < nunit; ++u) {
        const int r = u / npass, t0 = (u - r * npass) * 64;
        unit_idx(u + 2, jn2);
        if (u + 1 < nunit) {
            validate(jn);
            issue(u + 1, jn);
            unit_keys(jn, kn);
            dwn = unit_dout(u + 1);
            unit_q(u + 1, qn);
        }
        // dO_i in column 0 of B: lanes 0..3 take words 8 ks + t and 8 ks + t + 4
        uint32_t bd[4][2];
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            const uint32_t x0 = __shfl_sync(kFull, dwc, 8 * ks + s4);
            const uint32_t x1 = __shfl_sync(kFull, dwc, 8 * ks + s4 + 4);
            bd[ks][0] = g4 == 0 ? x0 : 0u;
            bd[ks][1] = g4 == 0 ? x1 : 0u;
        }
        if (u + 1 < nunit) cp_async_wait<1>();
        else cp_async_wait<0>();
        __syncwarp();
        const uint32_t slot = ring + (uint32_t)(u & 1) * slot_bytes;
        const int nmt = min(4, (k - t0 + 15) >> 4);      // 16-key tiles in this pass
        float cg[4][4];
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) cg[mt][e] = 0.f;
            if (mt < nmt) {
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    uint32_t af[4];
                    ldsm_x4(af, slot + (uint32_t)swz(16 * mt + (lane & 7) + 8 * ((lane >> 3) & 1),
                                                     2 * ks + (lane >> 4)) * 2u);
                    mma16816(cg[mt], af, bd[ks][0], bd[ks][1]);
                }
            }
        }
        __syncwarp();                            // slot reads done before it is refilled
        // slot L: tile L >> 4, row half (L >> 3) & 1, row L & 7 -> lane 4 (L & 7)
        float gown[2] = {0.f, 0.f};
        const int srcl = (lane & 7) * 4;
        const bool hi = (lane >> 3) & 1, up = lane >> 4;
#pragma unroll
        for (int sl = 0; sl < 2; ++sl) {
            if (2 * sl < nmt) {
                const float x0 = __shfl_sync(kFull, cg[2 * sl][0], srcl);
                const float x1 = __shfl_sync(kFull, cg[2 * sl][2], srcl);
                const float x2 = __shfl_sync(kFull, cg[2 * sl + 1][0], srcl);
                const float x3 = __shfl_sync(kFull, cg[2 * sl + 1][2], srcl);
                gown[sl] = up ? (hi ? x3 : x2) : (hi ? x1 : x0);
            }
        }
        float d2v[2];
#pragma unroll
        for (int s = 0; s < 2; ++s) d2v[s] = jc[s] >= 0 ? dist2k<DK>(qi, kc[s]) : INFINITY;
        if constexpr (WK == kWSoftmax) {
            float pm = fminf(d2v[0], d2v[1]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) pm = fminf(pm, __shfl_xor_sync(kFull, pm, o));
            const float mn = fminf(mrun, pm);
            if (mn != mrun) {                    // uniform across the warp
                if (mrun != INFINITY)
                    acc.rebase(dup2(mn - mrun), dup2(shift_scale(mn, mrun, inv_g2)), k2w);
                mrun = mn;
            }
        }
        {
            // empty slots: weight 0 and d2 = m, so that they add nothing (the shift
            // is still infinite only while every slot so far was empty)
            const bool v0 = jc[0] >= 0, v1 = jc[1] >= 0;
            const float mf = mrun == INFINITY ? 0.f : mrun;
            const float2 d2p = make_float2(v0 ? d2v[0] : mf, v1 ? d2v[1] : mf);
            const float2 mp = dup2(mf);
            float2 w = weight_fast2<WK>(d2p, mp, ig2w);
            w.x = v0 ? w.x : 0.f;
            w.y = v1 ? w.y : 0.f;
            const float kc0[4] = {kc[0].x, kc[0].y, kc[0].z, kc[0].w};
            const float kc1[4] = {kc[1].x, kc[1].y, kc[1].z, kc[1].w};
            float2 dqp[4];
#pragma unroll
            for (int d = 0; d < 4; ++d) dqp[d] = make_float2(qi[d] - kc0[d], qi[d] - kc1[d]);
            acc.add<DK, WK>(w, d2p, mp, make_float2(gown[0], gown[1]), dqp, m2ig2w, two_igw, k2w);
        }
        if (t0 + 64 >= k) {                      // the query's last pass: its window sums
            float tv[16];
#pragma unroll
            for (int y = 0; y < 16; ++y) tv[y] = y < 12 ? acc.x[y].x + acc.x[y].y : 0.f;
            const float tot = warp_transpose_sum16(tv, lane);      // value (lane >> 1)
            const int row = warp * 16 + r;
            if (!(lane & 1) && (lane >> 1) < 12) qpart[row][lane >> 1] = tot;
            if (lane == 0) qmpart[row] = mrun;
            acc.zero();
            mrun = INFINITY;
        }
        jc[0] = jn[0]; jc[1] = jn[1];
        jn[0] = jn2[0]; jn[1] = jn2[1];
        kc[0] = kn[0]; kc[1] = kn[1];
        dwc = dwn;
#pragma unroll
        for (int d = 0; d < 4; ++d) qi[d] = qn[d];
    }
    // every warp's walk is done before the rings become the own-chunk tiles
    __syncthreads();
    stage_rows(own.dO, db, i0, iend);
    load_ktile(0, cC);
    cp_async_commit();

    // ------------------------------------------------- own-chunk part ---
    const int g8 = lane >> 2, tig = lane & 3;
    const int ra = i0 + warp * 16 + g8, rb = ra + 8;
    float qa[4], qbv[4];
#pragma unroll
    for (int d = 0; d < 4; ++d) {
        qa[d] = (ra < iend && d < DK) ? qb[(int64_t)ra * DK + d] : 0.f;
        qbv[d] = (rb < iend && d < DK) ? qb[(int64_t)rb * DK + d] : 0.f;
    }
    const int lim_a = ra < iend ? ra : -1, lim_b = rb < iend ? rb : -1;
    const int warp_first = i0 + warp * 16;
    const int warp_last = min(warp_first + 15, iend - 1);
    const bool warp_rows_full = warp_first + 15 < iend;
    float2 qab[4];
#pragma unroll
    for (int d = 0; d < 4; ++d) qab[d] = make_float2(qa[d], qbv[d]);
    const float2 ig2 = dup2(inv_g2), m2ig2 = dup2(-2.f * inv_g2), two_ig = dup2(2.f * inv_g);
    const float2 k2v = dup2(k2);
    QAcc2 lab;
    lab.zero();
    uint32_t afr[4][4];
    const int rowa_l = warp * 16 + g8;
    float2 mab = make_float2(qmpart[rowa_l], qmpart[rowa_l + 8]);   // softmax shifts
    auto tile = [&](const float4 *Ks, uint32_t vbase, int key0, auto masked) {
        if constexpr (WK == kWSoftmax) {           // move the shift to this tile's minimum
            // (keys read through a volatile view: distances recomputed below are
            // not kept alive across the mma)
            const volatile float4 *Kv = Ks;
            float2 tmin = make_float2(INFINITY, INFINITY);
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int kl = nt * 8 + 2 * tig + e;
                    const float4 kv = make_float4(Kv[kl].x, Kv[kl].y, Kv[kl].z, Kv[kl].w);
                    const float kc[4] = {kv.x, kv.y, kv.z, kv.w};
                    float2 d2 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int d = 0; d < DK; ++d) {
                        const float2 t = sub2(qab[d], dup2(kc[d]));
                        d2 = fma2(t, t, d2);
                    }
                    if (decltype(masked)::value) {
                        const int key = key0 + kl;
                        d2.x = key <= lim_a ? d2.x : INFINITY;
                        d2.y = key <= lim_b ? d2.y : INFINITY;
                    }
                    tmin = make_float2(fminf(tmin.x, d2.x), fminf(tmin.y, d2.y));
                }
#pragma unroll
            for (int o = 1; o <= 2; o <<= 1) {
                tmin.x = fminf(tmin.x, __shfl_xor_sync(kFull, tmin.x, o));
                tmin.y = fminf(tmin.y, __shfl_xor_sync(kFull, tmin.y, o));
            }
            const float2 mn = make_float2(fminf(mab.x, tmin.x), fminf(mab.y, tmin.y));
            const float2 dm = make_float2(mab.x == INFINITY ? 0.f : mn.x - mab.x,
                                          mab.y == INFINITY ? 0.f : mn.y - mab.y);
            lab.rebase(dm, make_float2(shift_scale(mn.x, mab.x, inv_g2),
                                       shift_scale(mn.y, mab.y, inv_g2)), k2v);
            mab = mn;
        }
        float s[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[nt][e] = 0.f;
        const int m = lane >> 3, rr = lane & 7;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                const int key = np * 16 + (m >> 1) * 8 + rr;
                uint32_t b[4];
                ldsm_x4(b, vbase + (uint32_t)swz(key, ks * 2 + (m & 1)) * 2u);
                mma16816(s[2 * np], afr[ks], b[0], b[1]);
                mma16816(s[2 * np + 1], afr[ks], b[2], b[3]);
            }
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int kl = nt * 8 + 2 * tig + e;
                const float4 kv = Ks[kl];
                const float kc[4] = {kv.x, kv.y, kv.z, kv.w};
                float2 dq[4];
                float2 d2 = make_float2(0.f, 0.f);
#pragma unroll
                for (int d = 0; d < DK; ++d) {
                    dq[d] = sub2(qab[d], dup2(kc[d]));
                    d2 = fma2(dq[d], dq[d], d2);
                }
                float2 w = weight_fast2<WK>(d2, mab, ig2);
                if (decltype(masked)::value) {
                    const int key = key0 + kl;
                    w.x = key <= lim_a ? w.x : 0.f;
                    w.y = key <= lim_b ? w.y : 0.f;
                }
                lab.add<DK, WK>(w, d2, mab, make_float2(s[nt][e], s[nt][2 + e]), dq, m2ig2, two_ig,
                                k2v);
            }
    };
    for (int kt = 0; kt < nkt; ++kt) {
        if (kt + 1 < nkt) load_ktile((kt + 1) & 1, cC + (kt + 1) * T64);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        if (kt == 0) {
            const uint32_t dbase = smem_u32(own.dO);
            const int m = lane >> 3, rr = lane & 7;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const int row = warp * 16 + (m & 1) * 8 + rr;
                ldsm_x4(afr[ks], dbase + (uint32_t)swz(row, ks * 2 + (m >> 1)) * 2u);
            }
        }
        const int key0 = cC + kt * T64;
        if (key0 <= warp_last) {
            const float4 *Ks = own.kt[kt & 1];
            const uint32_t vbase = smem_u32(own.v[kt & 1]);
            if (warp_rows_full && key0 + T64 - 1 <= warp_first)
                tile(Ks, vbase, key0, std::false_type{});
            else
                tile(Ks, vbase, key0, std::true_type{});
        }
        __syncthreads();
    }
    QAcc la, lb;
#pragma unroll
    for (int y = 0; y < 12; ++y) {
        la.x[y] = lab.x[y].x;
        lb.x[y] = lab.x[y].y;
    }

    // ------------------------------------------------------- epilogue ---
#pragma unroll
    for (int y = 0; y < 12; ++y) {
        la.x[y] += __shfl_xor_sync(kFull, la.x[y], 1);
        la.x[y] += __shfl_xor_sync(kFull, la.x[y], 2);
        lb.x[y] += __shfl_xor_sync(kFull, lb.x[y], 1);
        lb.x[y] += __shfl_xor_sync(kFull, lb.x[y], 2);
    }
    if (tig < 2) {
        const int rloc = warp * 16 + g8 + tig * 8;
        const int i = i0 + rloc;
        if (i < iend) {
            QAcc wpart;                            // the window part, on the final shift
#pragma unroll
            for (int y = 0; y < 12; ++y) wpart.x[y] = qpart[rloc][y];
            const float mfin = tig == 0 ? mab.x : mab.y;
            if constexpr (WK == kWSoftmax) {
                const float mw = qmpart[rloc];
                if (mw != INFINITY) wpart.rebase(mfin - mw, shift_scale(mfin, mw, inv_g2), k2);
            }
            float t[12];
#pragma unroll
            for (int y = 0; y < 12; ++y) t[y] = (tig == 0 ? la.x[y] : lb.x[y]) + wpart.x[y];
            const float inv_s = __frcp_rn(t[0]);
            const float gb = t[1] * inv_s;
            const int64_t gi = seg * N + i;
            if constexpr (WK == kWCauchy) {
                // dq_d = -2/gamma^2 (sum u g (q-k)_d - gbar sum u (q-k)_d) / s and
                // dgamma_i = 2/gamma (sum g w - sum g u - gbar (sum w - sum u)) / s
                //          = 2/gamma (gbar sum u - sum u g) / s   (sum g w = gbar s)
                const float cq = -2.f * inv_g2 * inv_s, cg = 2.f * inv_g * inv_s;
                for (int d = 0; d < DK; ++d)
                    dq[gi * DK + d] = (t[4 + d] - gb * t[8 + d]) * cq;
                dg_part[gi] = (gb * t[3] - t[2]) * cg;
            } else {
                for (int d = 0; d < DK; ++d) dq[gi * DK + d] = (t[4 + d] - gb * t[8 + d]) * inv_s;
                dg_part[gi] = (t[2] - gb * t[3]) * inv_s;
            }
            const float *qq = tig == 0 ? qa : qbv;
            QRec rcd;
            rcd.q = make_float4(qq[0], qq[1], qq[2], qq[3]);
            rcd.sg = make_float4(inv_s, -gb * inv_s, WK == kWSoftmax ? mfin : 0.f, gb);
            rec[gi] = rcd;
        }
    }
}

// ============================================================== key side ===

// Tiles of the own-chunk part.  A query tile's records are staged 48 bytes
// apart (the 32-byte record and 16 bytes of padding): the four records a
// quarter-warp reads at once then start in four different bank groups, where a
// 32- or 64-byte stride puts two of them on the same banks.
constexpr int kRecPad = 3;                        // float4 slots per staged record
struct __align__(16) KOwn {
    __nv_bfloat16 v[T64 * DV];
    __nv_bfloat16 dO[2][T64 * DV];
    float4 qr[2][T64][kRecPad];
};
constexpr int kKeyWarps = THREADS / 32;
constexpr uint32_t kRingBytes = 2 * 32 * DV * 2;   // one warp's two slots of 32 dO rows
constexpr int kGs = 24;                            // row stride (floats) of the G scratch
// Column swizzle of the G scratch (even, so float2 pairs stay together): the
// read of one column by all 32 rows spreads over 16 banks instead of 4.
__device__ __forceinline__ int gs_swz(int row) { return ((row >> 2) & 3) << 1; }
constexpr size_t kKeyBig = sizeof(KOwn) > kKeyWarps * kRingBytes ? sizeof(KOwn)
                                                                 : kKeyWarps * kRingBytes;

// The window walk's rings and the own-chunk tiles share `big` (the walk ends in
// every warp before the tiles are staged); a warp's G scratch lives in its own
// rows of dvp until its dv rows are written there.
struct __align__(16) KSmem {
    unsigned char big[kKeyBig];
    float dvp[T64][DV + 4];
    float dkp[T64][4];
};
static_assert(32 * kGs <= 16 * (DV + 4), "G scratch fits in a warp's dvp rows");

template <int DK, int WK>
__global__ void __launch_bounds__(THREADS, 4)
bwd_key_tc(const float *__restrict__ kx, const __nv_bfloat16 *__restrict__ v,
           const float *__restrict__ gamma, const __nv_bfloat16 *__restrict__ dout,
           const QRec *__restrict__ rec, const uint32_t *__restrict__ csr_q,
           const uint32_t *__restrict__ csr_k, uint32_t csr_mask, int kgs,
           const uint32_t *__restrict__ off, int64_t csr_stride, float *__restrict__ dk,
           __nv_bfloat16 *__restrict__ dv, const float *__restrict__ own_dv,
           const float *__restrict__ own_dk, int N, int H, int C, int tiles_per_chunk) {
    extern __shared__ __align__(16) unsigned char key_smem[];
    KSmem &sm = *reinterpret_cast<KSmem *>(key_smem);
    KOwn &own = *reinterpret_cast<KOwn *>(sm.big);
    const int64_t seg = blockIdx.y;
    const int c = blockIdx.x / tiles_per_chunk;
    const int kt = blockIdx.x % tiles_per_chunk;
    const int cC = c * C, cend = cC + C;
    const int j0 = cC + kt * T64;
    const int jend = min(cend, j0 + T64);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float gm = gamma[seg % H];
    const float inv_g2 = __frcp_rn(gm * gm);
    const float *kb = kx + seg * (int64_t)N * DK;
    const __nv_bfloat16 *vb = v + seg * (int64_t)N * DV;
    const __nv_bfloat16 *db = dout + seg * (int64_t)N * DV;
    const QRec *rb_ = rec + seg * (int64_t)N;

    auto load_qtile = [&](int b, int iq0) {
        stage_rows(own.dO[b], db, iq0, cend);
        if (threadIdx.x < T64 * 2) {
            const int r = threadIdx.x >> 1, h = threadIdx.x & 1;
            const int i = iq0 + r;
            const bool ok = i < cend;
            cp_async16(smem_u32(&own.qr[b][r][h]),
                       reinterpret_cast<const float4 *>(rb_ + (ok ? i : iq0)) + h, ok ? 16 : 0);
        }
    };
    // ---------------------------------------------------- window part ---
    // The queries that selected this warp's 16 keys are one contiguous run of
    // the transposed lists, walked 32 entries at a time whatever key each entry
    // belongs to (the run need not be ordered by key).  Lane e owns entry e of a
    // step: its key (from the list word, or the key array of the unpacked
    // lists), its query's record, w, a = w / s and the dk term.  The step's 32
    // dO rows are copied into a two-slot ring of swizzled 128-byte rows in
    // shared memory (cp.async) one step ahead, the list entries two steps ahead.
    // With the 16 keys' v rows as the columns of B, G = dO_rows . V_keys^T on
    // the tensor cores gives every entry's g in the column of its key (read
    // back through a small scratch tile), and dV_keys += dO^T A, A holding a in
    // the column of the entry's key, accumulates all 16 keys' dv in the mma
    // registers over the whole walk.  A key half (8 columns) that no entry of a
    // 16-entry tile belongs to is skipped.  dk is summed per key on the tensor
    // cores too: dk_keys += OneHot^T X, X holding each entry's dk term split
    // into a bf16 high part and a bf16 remainder (8 columns: d_K <= 4 dims x 2),
    // staged as one 16-byte row per entry and read back by a transposing
    // ldmatrix; the two parts are added at the end.
    const uint32_t *lst = csr_q + seg * csr_stride;
    const uint32_t *klst = csr_k ? csr_k + seg * csr_stride : nullptr;
    // list offsets per key (kgs = 0) or per 8-key group (kgs = 3: a warp's 16
    // keys are then two groups)
    const uint32_t *ob = off + seg * (int64_t)((N >> kgs) + 1);
    constexpr uint32_t kNone = 0xffffffffu;
    const int wj0 = j0 + warp * 16;
    const int nkw = max(0, min(16, jend - wj0));
    const uint32_t P0 = nkw > 0 ? ob[wj0 >> kgs] : 0u;
    const uint32_t P1 = nkw > 0 ? ob[(wj0 + nkw) >> kgs] : 0u;
    const int nch = nkw > 0 ? (int)((P1 - P0 + 31) >> 5) : 0;
    const int g4 = lane >> 2, s4 = lane & 3;
    float kc[4] = {0.f, 0.f, 0.f, 0.f};                       // lane r: key r's coordinates
    if (lane < nkw) {
        const float4 t = load_k4(kb + (int64_t)(wj0 + lane) * DK, DK);
        kc[0] = t.x; kc[1] = t.y; kc[2] = t.z; kc[3] = t.w;
    }
    // B fragments of G: column g of key half h is v of key 8h + g; rows are the
    // dimensions 16 ks + 2t, +1 and 16 ks + 2t + 8, +9
    uint32_t vbf[2][4][2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int key = 8 * h + g4;
        const uint32_t *vr = reinterpret_cast<const uint32_t *>(vb + (int64_t)(wj0 + key) * DV);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            vbf[h][ks][0] = key < nkw ? vr[8 * ks + s4] : 0u;
            vbf[h][ks][1] = key < nkw ? vr[8 * ks + s4 + 4] : 0u;
        }
    }
    float cdv[4][2][4];          // dv of the 16 keys: dims 16c + g (+8) x keys 8h + 2t (+1)
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int e = 0; e < 4; ++e) cdv[c][h][e] = 0.f;
    float cdk[4] = {0.f, 0.f, 0.f, 0.f};   // dk: keys g (+8) x columns 2t, 2t+1 (hi 0-3, lo 4-7)
    const uint32_t ring = smem_u32(sm.big) + (uint32_t)warp * kRingBytes;
    float *gs = &sm.dvp[warp * 16][0];                        // G scratch: [32 entries][kGs]
    const uint32_t gsa = smem_u32(gs);                        // ... then the dk rows [32][8] bf16
    // entry n*32 + lane of the run: its query (kNone past the end) and its key
    auto list_at = [&](int n, uint32_t &ie, int &kr) {
        const uint32_t pp = P0 + 32u * (uint32_t)n + (uint32_t)lane;
        ie = kNone;
        kr = 0;
        if (n < nch && pp < P1) {
            const uint32_t wd = __ldg(lst + pp);
            ie = wd & csr_mask;
            kr = (int)(klst ? __ldg(klst + pp) : (wd >> 16)) - wj0;
        }
    };
    auto issue = [&](int n, uint32_t ie) {                    // dO rows of step n
        const uint32_t slot = ring + (uint32_t)(n & 1) * (kRingBytes / 2);
#pragma unroll
        for (int h = 0; h < 8; ++h) {
            const int row = 4 * h + (lane >> 3), ch = lane & 7;
            const uint32_t iu = __shfl_sync(kFull, ie, row);
            const bool ok = iu != kNone;
            cp_async16(slot + (uint32_t)swz(row, ch) * 2u, db + (int64_t)(ok ? iu : 0u) * DV + ch * 8,
                       ok ? 16 : 0);
        }
        cp_async_commit();
    };
    auto record = [&](uint32_t ie, float4 &r0, float4 &r1) {
        if (ie != kNone) {
            const float4 *src = reinterpret_cast<const float4 *>(rb_ + ie);
            r0 = __ldg(src);
            r1 = __ldg(src + 1);
        } else {
            r0 = make_float4(0.f, 0.f, 0.f, 0.f);
            r1 = r0;
        }
    };
    uint32_t ie_cur, ie_nxt;
    int kr_cur, kr_nxt;
    list_at(0, ie_cur, kr_cur);
    float4 rn0, rn1;
    if (nch > 0) issue(0, ie_cur);
    record(ie_cur, rn0, rn1);
    list_at(1, ie_nxt, kr_nxt);
    for (int n = 0; n < nch; ++n) {
        const float4 rq0 = rn0, rq1 = rn1;
        const uint32_t ie = ie_cur;
        const int kr = kr_cur;
        if (n + 1 < nch) {
            issue(n + 1, ie_nxt);
            record(ie_nxt, rn0, rn1);
        }
        ie_cur = ie_nxt;
        kr_cur = kr_nxt;
        list_at(n + 2, ie_nxt, kr_nxt);
        if (n + 1 < nch) cp_async_wait<1>();
        else cp_async_wait<0>();
        __syncwarp();
        const uint32_t slot = ring + (uint32_t)(n & 1) * (kRingBytes / 2);
        const uint32_t base = P0 + 32u * (uint32_t)n;
        const bool valid = ie != kNone;
        float kj[4];
#pragma unroll
        for (int d = 0; d < DK; ++d) kj[d] = __shfl_sync(kFull, kc[d], kr);
        float a = 0.f, s2 = 0.f, inv_s = 0.f, ngbs = 0.f;
        float dqk[4] = {0.f, 0.f, 0.f, 0.f};
        if (valid) {
            const float qc[4] = {rq0.x, rq0.y, rq0.z, rq0.w};
            float d2 = 0.f;
#pragma unroll
            for (int d = 0; d < DK; ++d) {
                dqk[d] = qc[d] - kj[d];
                d2 = __fmaf_rn(dqk[d], dqk[d], d2);
            }
            const float w = weight_fast<WK>(d2, rq1.z, inv_g2);
            inv_s = rq1.x;
            ngbs = rq1.y;
            a = w * inv_s;
            // Cauchy: 2 w^2 / gamma^2 with the constant applied to dk at the end
            s2 = WK == kWCauchy ? w * w : 2.f * neg_dw_dd2<WK>(w, inv_g2);
        }
        // key halves met by each 16-entry tile
        const int last = min(31, (int)(P1 - base) - 1);
        const unsigned blo = __ballot_sync(kFull, valid && kr < 8);
        const unsigned bhi = __ballot_sync(kFull, valid && kr >= 8);
        const uint32_t pk = ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a)) << 16) |
                            (uint32_t)kr;
        uint32_t ev[2][4];                                    // pk of entries 2t, 2t+1, 2t+8, 2t+9
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
            if (mt == 1 && last < 16) break;
            const bool half[2] = {((blo >> (16 * mt)) & 0xffffu) != 0u,
                                  ((bhi >> (16 * mt)) & 0xffffu) != 0u};
            uint32_t af[4][4];
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                ldsm_x4(af[ks], slot + (uint32_t)swz(16 * mt + (lane & 7) + 8 * ((lane >> 3) & 1),
                                                    2 * ks + (lane >> 4)) * 2u);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (!half[h]) continue;
                float cg[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) mma16816(cg, af[ks], vbf[h][ks][0], vbf[h][ks][1]);
                const int ra = 16 * mt + g4, rb2 = ra + 8;
                *reinterpret_cast<float2 *>(gs + ra * kGs + ((8 * h + 2 * s4) ^ gs_swz(ra))) =
                    make_float2(cg[0], cg[1]);
                *reinterpret_cast<float2 *>(gs + rb2 * kGs + ((8 * h + 2 * s4) ^ gs_swz(rb2))) =
                    make_float2(cg[2], cg[3]);
            }
            // dV_keys += dO^T A: entries 2t, 2t+1 (+8) of the tile in the rows of B
            ev[mt][0] = __shfl_sync(kFull, pk, 16 * mt + 2 * s4);
            ev[mt][1] = __shfl_sync(kFull, pk, 16 * mt + 2 * s4 + 1);
            ev[mt][2] = __shfl_sync(kFull, pk, 16 * mt + 2 * s4 + 8);
            ev[mt][3] = __shfl_sync(kFull, pk, 16 * mt + 2 * s4 + 9);
            // A of dim block c: the 8x8 blocks of the G fragments transposed in
            // registers (entries 0-7 | 8-15 x dims 0-7 | 8-15 of the block)
            uint32_t at[4][4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                at[c][0] = movmatrix_trans(af[c][0]);
                at[c][1] = movmatrix_trans(af[c][2]);
                at[c][2] = movmatrix_trans(af[c][1]);
                at[c][3] = movmatrix_trans(af[c][3]);
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (!half[h]) continue;
                const uint32_t key = (uint32_t)(8 * h + g4);
                auto pick = [key](uint32_t e) { return (e & 0xffffu) == key ? (e >> 16) : 0u; };
                const uint32_t b0 = pick(ev[mt][0]) | (pick(ev[mt][1]) << 16);
                const uint32_t b1 = pick(ev[mt][2]) | (pick(ev[mt][3]) << 16);
#pragma unroll
                for (int c = 0; c < 4; ++c) mma16816(cdv[c][h], at[c], b0, b1);
            }
        }
        __syncwarp();
        const float gown = valid ? gs[lane * kGs + (kr ^ gs_swz(lane))] : 0.f;
        const float coef = valid ? __fmaf_rn(gown, inv_s, ngbs) * s2 : 0.f;
        // this entry's dk term as a bf16 high part and remainder, one 16-byte row
        uint32_t xw[4];
#pragma unroll
        for (int hp = 0; hp < 2; ++hp) {
            float x[2], r[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int d = 2 * hp + e;
                x[e] = d < DK ? coef * dqk[d] : 0.f;
                r[e] = x[e] - __bfloat162float(__float2bfloat16_rn(x[e]));
            }
            xw[hp] = pack_bf16(x[0], x[1]);
            xw[2 + hp] = pack_bf16(r[0], r[1]);
        }
        __syncwarp();                            // G scratch read before the rows overwrite it
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(gsa + 16u * lane),
                     "r"(xw[0]), "r"(xw[1]), "r"(xw[2]), "r"(xw[3])
                     : "memory");
        __syncwarp();
        uint32_t bx[4];                          // B fragments: tile 0 entries 0-7 | 8-15, tile 1 ..
        ldsm_x4_trans(bx, gsa + 16u * lane);
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
            if (mt == 1 && last < 16) break;
            auto one = [](uint32_t e, int key) { return (int)(e & 0xffffu) == key ? 0x3F80u : 0u; };
            uint32_t ao[4];
            ao[0] = one(ev[mt][0], g4) | (one(ev[mt][1], g4) << 16);
            ao[1] = one(ev[mt][0], g4 + 8) | (one(ev[mt][1], g4 + 8) << 16);
            ao[2] = one(ev[mt][2], g4) | (one(ev[mt][3], g4) << 16);
            ao[3] = one(ev[mt][2], g4 + 8) | (one(ev[mt][3], g4 + 8) << 16);
            mma16816(cdk, ao, bx[2 * mt], bx[2 * mt + 1]);
        }
        __syncwarp();
    }
    // this warp's dv and dk rows (keys 8h + 2t (+1), dims 16c + g (+8))
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int row = warp * 16 + 8 * h + 2 * s4;
            const int col = 16 * c + g4;
            sm.dvp[row][col] = cdv[c][h][0];
            sm.dvp[row + 1][col] = cdv[c][h][1];
            sm.dvp[row][col + 8] = cdv[c][h][2];
            sm.dvp[row + 1][col + 8] = cdv[c][h][3];
        }
    // dk: the high parts (columns 0-3) and remainders (4-7) added; lane (g, t)
    // for t < 2 holds dims 2t, 2t+1 of keys g and g + 8
#pragma unroll
    for (int e = 0; e < 4; ++e) cdk[e] += __shfl_xor_sync(kFull, cdk[e], 2);
    if (s4 < 2) {
        *reinterpret_cast<float2 *>(&sm.dkp[warp * 16 + g4][2 * s4]) = make_float2(cdk[0], cdk[1]);
        *reinterpret_cast<float2 *>(&sm.dkp[warp * 16 + g4 + 8][2 * s4]) = make_float2(cdk[2], cdk[3]);
    }
    // every warp's walk is done before the rings become the own-chunk tiles
    __syncthreads();
    // (own_dv set: the own-chunk sums come from a separate kernel)
    if (!own_dv) {
        stage_rows(own.v, vb, j0, jend);
        load_qtile(0, j0);            // query tiles start at the key tile
        cp_async_commit();
    }

    // ------------------------------------------------- own-chunk part ---
    const int g8 = lane >> 2, tig = lane & 3;
    const int ka = j0 + warp * 16 + g8, kbi = ka + 8;      // this thread's two key rows
    const float4 kva = ka < jend ? load_k4(kb + (int64_t)ka * DK, DK) : make_float4(0, 0, 0, 0);
    const float4 kvb = kbi < jend ? load_k4(kb + (int64_t)kbi * DK, DK) : make_float4(0, 0, 0, 0);
    float2 kab[4];                                        // (row a, row b) coordinates
    kab[0] = make_float2(kva.x, kvb.x);
    kab[1] = make_float2(kva.y, kvb.y);
    kab[2] = make_float2(kva.z, kvb.z);
    kab[3] = make_float2(kva.w, kvb.w);
    const int first_a = ka < jend ? ka : 0x7fffffff;     // first query index row a may see
    const int first_b = kbi < jend ? kbi : 0x7fffffff;
    const float2 ig2 = dup2(inv_g2), two_ig2 = dup2(2.f * inv_g2);
    float dva[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) dva[nt][e] = 0.f;
    float2 dkab[4];
#pragma unroll
    for (int d = 0; d < 4; ++d) dkab[d] = make_float2(0.f, 0.f);
    const int nqt = tiles_per_chunk - kt;
    const int m = lane >> 3, rr = lane & 7;
    // every key row of this warp sees every query of a query tile starting at
    // or after its last key (within the chunk): no mask needed there
    const int warp_key_last = j0 + warp * 16 + 15;
    const bool warp_keys_full = warp_key_last < jend;
    // A of S^T: this warp's 16 key rows of V, loaded once the tiles are staged
    uint32_t va[4][4];
    auto qtile = [&](int t, int iq0, auto masked) {
        const uint32_t dbase = smem_u32(own.dO[t & 1]);
        const float4 (*qt_rec)[kRecPad] = own.qr[t & 1];
        // per 16 queries: S^T = V . dO^T (16 keys x 16 queries), the element-wise
        // terms for key rows (a, b) packed, P^T into A fragments, then
        // dV += P^T . dO with the same dO fragments transposed in registers
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            uint32_t bq[4][4];     // queries 16 kk + (0-7 | 8-15) x dims 16 ks + (0-7 | 8-15)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                ldsm_x4(bq[ks], dbase + (uint32_t)swz(kk * 16 + (m >> 1) * 8 + rr,
                                                     ks * 2 + (m & 1)) * 2u);
            float s[2][4];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                for (int e = 0; e < 4; ++e) s[hh][e] = 0.f;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                mma16816(s[0], va[ks], bq[ks][0], bq[ks][1]);
                mma16816(s[1], va[ks], bq[ks][2], bq[ks][3]);
            }
            float pa_[8];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int nt = 2 * kk + hh;
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int ql = nt * 8 + 2 * tig + e;
                    const float4 qv = qt_rec[ql][0];
                    const float qc[4] = {qv.x, qv.y, qv.z, qv.w};
                    float2 sgv;                    // (1/s, -gbar/s)
                    float mz = 0.f;                // softmax shift
                    if constexpr (WK == kWSoftmax) {
                        const float4 t4 = qt_rec[ql][1];
                        sgv = make_float2(t4.x, t4.y);
                        mz = t4.z;
                    } else {
                        sgv = *reinterpret_cast<const float2 *>(&qt_rec[ql][1]);
                    }
                    const float2 inv_s = dup2(sgv.x), ngbs = dup2(sgv.y);
                    const float2 mq = dup2(mz);
                    float2 dqk[4];
                    float2 d2 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int d = 0; d < DK; ++d) {
                        dqk[d] = sub2(dup2(qc[d]), kab[d]);
                        d2 = fma2(dqk[d], dqk[d], d2);
                    }
                    float2 w = weight_fast2<WK>(d2, mq, ig2);
                    if (decltype(masked)::value) {
                        const int i = iq0 + ql;
                        w.x = (i >= first_a && i < cend) ? w.x : 0.f;
                        w.y = (i >= first_b && i < cend) ? w.y : 0.f;
                    }
                    const float2 aw = mul2(w, inv_s);
                    const float2 dldw = fma2(make_float2(s[hh][e], s[hh][2 + e]), inv_s, ngbs);
                    float2 ndw;                    // 2 (-dw/d(d^2))
                    if constexpr (WK == kWSoftmax) ndw = mul2(w, two_ig2);
                    else if constexpr (WK == kWInvEuclid) ndw = mul2(mul2(w, w), w);
                    else ndw = mul2(w, w);         // 2/gamma^2 applied to dk at the end
                    const float2 coef = mul2(dldw, ndw);
#pragma unroll
                    for (int d = 0; d < DK; ++d) dkab[d] = fma2(coef, dqk[d], dkab[d]);
                    pa_[hh * 4 + e] = aw.x;
                    pa_[hh * 4 + 2 + e] = aw.y;
                }
            }
            uint32_t pa[4];
            pa[0] = pack_bf16(pa_[0], pa_[1]);     // key row g,   queries 2tig..+1
            pa[1] = pack_bf16(pa_[2], pa_[3]);     // key row g+8
            pa[2] = pack_bf16(pa_[4], pa_[5]);     // key row g,   queries +8
            pa[3] = pack_bf16(pa_[6], pa_[7]);     // key row g+8, queries +8
#pragma unroll
            for (int np = 0; np < 4; ++np) {       // dims 16 np + (0-7 | 8-15)
                mma16816(dva[2 * np], pa, movmatrix_trans(bq[np][0]), movmatrix_trans(bq[np][2]));
                mma16816(dva[2 * np + 1], pa, movmatrix_trans(bq[np][1]),
                         movmatrix_trans(bq[np][3]));
            }
        }
    };
    for (int t = 0; t < (own_dv ? 0 : nqt); ++t) {
        const int iq0 = j0 + t * T64;
        if (t + 1 < nqt) load_qtile((t + 1) & 1, iq0 + T64);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        if (t == 0) {
            const uint32_t vbase = smem_u32(own.v);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                ldsm_x4(va[ks], vbase + (uint32_t)swz(warp * 16 + (m & 1) * 8 + rr,
                                                     ks * 2 + (m >> 1)) * 2u);
        }
        if (warp_keys_full && iq0 >= warp_key_last && iq0 + T64 <= cend)
            qtile(t, iq0, std::false_type{});
        else
            qtile(t, iq0, std::true_type{});
        __syncthreads();
    }
    float dkl_a[4], dkl_b[4];
#pragma unroll
    for (int d = 0; d < 4; ++d) {
        dkl_a[d] = dkab[d].x;
        dkl_b[d] = dkab[d].y;
    }

    // ------------------------------------------------------- epilogue ---
#pragma unroll
    for (int d = 0; d < 4; ++d) {
        dkl_a[d] += __shfl_xor_sync(kFull, dkl_a[d], 1);
        dkl_a[d] += __shfl_xor_sync(kFull, dkl_a[d], 2);
        dkl_b[d] += __shfl_xor_sync(kFull, dkl_b[d], 1);
        dkl_b[d] += __shfl_xor_sync(kFull, dkl_b[d], 2);
    }
    const int rowa = warp * 16 + g8, rowb = rowa + 8;
    if (own_dv) {                    // the separate kernel's own-chunk sums
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            const int col = nt * 8 + 2 * tig;
            const float2 oa = ka < jend ? *reinterpret_cast<const float2 *>(
                                              own_dv + (seg * N + ka) * (int64_t)DV + col)
                                        : dup2(0.f);
            const float2 ob = kbi < jend ? *reinterpret_cast<const float2 *>(
                                               own_dv + (seg * N + kbi) * (int64_t)DV + col)
                                         : dup2(0.f);
            dva[nt][0] = oa.x;
            dva[nt][1] = oa.y;
            dva[nt][2] = ob.x;
            dva[nt][3] = ob.y;
        }
        if (tig == 0) {
#pragma unroll
            for (int d = 0; d < DK; ++d) {
                dkl_a[d] = ka < jend ? own_dk[(seg * N + ka) * 4 + d] : 0.f;
                dkl_b[d] = kbi < jend ? own_dk[(seg * N + kbi) * 4 + d] : 0.f;
            }
        }
    }
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
        const int col = nt * 8 + 2 * tig;
        if (ka < jend) {
            const float o0 = dva[nt][0] + sm.dvp[rowa][col];
            const float o1 = dva[nt][1] + sm.dvp[rowa][col + 1];
            *reinterpret_cast<__nv_bfloat162 *>(dv + (seg * N + ka) * (int64_t)DV + col) =
                __floats2bfloat162_rn(o0, o1);
        }
        if (kbi < jend) {
            const float o0 = dva[nt][2] + sm.dvp[rowb][col];
            const float o1 = dva[nt][3] + sm.dvp[rowb][col + 1];
            *reinterpret_cast<__nv_bfloat162 *>(dv + (seg * N + kbi) * (int64_t)DV + col) =
                __floats2bfloat162_rn(o0, o1);
        }
    }
    if (tig == 0) {
        const float ks = WK == kWCauchy ? 2.f * inv_g2 : 1.f;   // the Cauchy terms' constant
        for (int d = 0; d < DK; ++d) {
            if (ka < jend) dk[(seg * N + ka) * DK + d] = (dkl_a[d] + sm.dkp[rowa][d]) * ks;
            if (kbi < jend) dk[(seg * N + kbi) * DK + d] = (dkl_b[d] + sm.dkp[rowb][d]) * ks;
        }
    }
}

}  // namespace

bool attend_bwd_tc_supported(const Prob &p) {
    return p.vdt == ZETA_BF16 && p.dV == DV && p.dK <= 4;
}

size_t bwd_tc_rec_bytes(const Prob &p) { return sizeof(QRec) * (size_t)(p.S * p.N); }

template <int D, int WK>
cudaError_t bwd_query_tc_launch(const Prob &p, dim3 grid, int tpc, const float *q, const float *k,
                                const void *v, const float *gamma, const int32_t *idx,
                                const void *dout, float *dq, void *rec, float *dg_part,
                                int32_t *status, cudaStream_t st) {
    static PerDeviceOnce smem_once;          // run once per device, outside any capture
    const cudaError_t e = smem_once.run([] {  // the largest ring (k >= 64)
        return cudaFuncSetAttribute(bwd_query_tc<D, WK>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)q_smem_bytes(64));
    });
    if (e != cudaSuccess) return e;
    bwd_query_tc<D, WK><<<grid, THREADS, q_smem_bytes(p.k), st>>>(
        q, k, static_cast<const __nv_bfloat16 *>(v), gamma, idx,
        static_cast<const __nv_bfloat16 *>(dout), dq, static_cast<QRec *>(rec), dg_part, status,
        p.N, p.H, p.k, p.C, tpc);
    return cudaGetLastError();
}

template <int WK>
cudaError_t bwd_query_tc_dk(const Prob &p, dim3 grid, int tpc, const float *q, const float *k,
                            const void *v, const float *gamma, const int32_t *idx,
                            const void *dout, float *dq, void *rec, float *dg_part,
                            int32_t *status, cudaStream_t st) {
    switch (p.dK) {
        case 1: return bwd_query_tc_launch<1, WK>(p, grid, tpc, q, k, v, gamma, idx, dout, dq,
                                                  rec, dg_part, status, st);
        case 2: return bwd_query_tc_launch<2, WK>(p, grid, tpc, q, k, v, gamma, idx, dout, dq,
                                                  rec, dg_part, status, st);
        case 3: return bwd_query_tc_launch<3, WK>(p, grid, tpc, q, k, v, gamma, idx, dout, dq,
                                                  rec, dg_part, status, st);
        default: return bwd_query_tc_launch<4, WK>(p, grid, tpc, q, k, v, gamma, idx, dout, dq,
                                                   rec, dg_part, status, st);
    }
}

template <int D, int WK>
cudaError_t bwd_key_tc_launch(const Prob &p, dim3 grid, int tpc, const float *k, const void *v,
                              const float *gamma, const void *dout, const void *rec,
                              const uint32_t *csr_q, const uint32_t *csr_k, uint32_t csr_mask,
                              int kgs, const uint32_t *off,
                              int64_t csr_stride, float *dk, void *dv, const float *own_dv,
                              const float *own_dk, cudaStream_t st) {
    static PerDeviceOnce smem_once;          // run once per device, outside any capture
    const cudaError_t e = smem_once.run([] {
        return cudaFuncSetAttribute(bwd_key_tc<D, WK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)sizeof(KSmem));
    });
    if (e != cudaSuccess) return e;
    bwd_key_tc<D, WK><<<grid, THREADS, sizeof(KSmem), st>>>(
        k, static_cast<const __nv_bfloat16 *>(v), gamma, static_cast<const __nv_bfloat16 *>(dout),
        static_cast<const QRec *>(rec), csr_q, csr_k, csr_mask, kgs, off, csr_stride, dk,
        static_cast<__nv_bfloat16 *>(dv), own_dv, own_dk, p.N, p.H, p.C, tpc);
    return cudaGetLastError();
}

template <int WK>
cudaError_t bwd_key_tc_dk(const Prob &p, dim3 grid, int tpc, const float *k, const void *v,
                          const float *gamma, const void *dout, const void *rec,
                          const uint32_t *csr_q, const uint32_t *csr_k, uint32_t csr_mask,
                          int kgs, const uint32_t *off, int64_t csr_stride, float *dk, void *dv,
                          const float *own_dv, const float *own_dk, cudaStream_t st) {
    switch (p.dK) {
        case 1: return bwd_key_tc_launch<1, WK>(p, grid, tpc, k, v, gamma, dout, rec, csr_q, csr_k,
                                                csr_mask, kgs, off, csr_stride, dk, dv, own_dv,
                                                own_dk, st);
        case 2: return bwd_key_tc_launch<2, WK>(p, grid, tpc, k, v, gamma, dout, rec, csr_q, csr_k,
                                                csr_mask, kgs, off, csr_stride, dk, dv, own_dv,
                                                own_dk, st);
        case 3: return bwd_key_tc_launch<3, WK>(p, grid, tpc, k, v, gamma, dout, rec, csr_q, csr_k,
                                                csr_mask, kgs, off, csr_stride, dk, dv, own_dv,
                                                own_dk, st);
        default: return bwd_key_tc_launch<4, WK>(p, grid, tpc, k, v, gamma, dout, rec, csr_q, csr_k,
                                                 csr_mask, kgs, off, csr_stride, dk, dv, own_dv,
                                                 own_dk, st);
    }
}

cudaError_t launch_bwd_query_tc(const Prob &p, const float *q, const float *k, const void *v,
                                const float *gamma, const int32_t *idx, const void *dout,
                                float *dq, void *rec, float *dg_part, int32_t *status,
                                cudaStream_t st) {
    const int tpc = (p.C + T64 - 1) / T64;
    const dim3 grid((unsigned)(p.n * tpc), (unsigned)p.S);
    if (p.wk == kWSoftmax)
        return bwd_query_tc_dk<kWSoftmax>(p, grid, tpc, q, k, v, gamma, idx, dout, dq, rec,
                                          dg_part, status, st);
    if (p.wk == kWInvEuclid)
        return bwd_query_tc_dk<kWInvEuclid>(p, grid, tpc, q, k, v, gamma, idx, dout, dq, rec,
                                            dg_part, status, st);
    return bwd_query_tc_dk<kWCauchy>(p, grid, tpc, q, k, v, gamma, idx, dout, dq, rec, dg_part,
                                     status, st);
}

cudaError_t launch_bwd_key_tc(const Prob &p, const float *k, const void *v, const float *gamma,
                              const void *dout, const void *rec, const uint32_t *csr_q,
                              const uint32_t *csr_k, uint32_t csr_mask, int kgs,
                              const uint32_t *off, int64_t csr_stride,
                              float *dk, void *dv, const float *own_dv, const float *own_dk,
                              cudaStream_t st) {
    const int tpc = (p.C + T64 - 1) / T64;
    const dim3 grid((unsigned)(p.n * tpc), (unsigned)p.S);
    if (p.wk == kWSoftmax)
        return bwd_key_tc_dk<kWSoftmax>(p, grid, tpc, k, v, gamma, dout, rec, csr_q, csr_k,
                                        csr_mask, kgs,
                                        off, csr_stride, dk, dv, own_dv, own_dk, st);
    if (p.wk == kWInvEuclid)
        return bwd_key_tc_dk<kWInvEuclid>(p, grid, tpc, k, v, gamma, dout, rec, csr_q, csr_k,
                                          csr_mask, kgs,
                                          off, csr_stride, dk, dv, own_dv, own_dk, st);
    return bwd_key_tc_dk<kWCauchy>(p, grid, tpc, k, v, gamma, dout, rec, csr_q, csr_k, csr_mask,
                                   kgs, off,
                                   csr_stride, dk, dv, own_dv, own_dk, st);
}

}  // namespace zeta
