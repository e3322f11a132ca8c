// curves.cu -- the union of one window per Z-order curve (the axis-permuted
// codes themselves come from encode.cu).
//
// Passage: OpenReview discussion of "ZETA: Leveraging Z-order Curves for
// Efficient Top-k Attention", follow-up reply on interleaving the bits of
// different dimensions (several curves): the
// coordinates of each key are interleaved in several orders (the three cyclic
// shifts of (K^1, K^2, K^3), or all six orderings) and every curve contributes
// k // curves of the k selected tokens.
//
// Reading of the union: windows are listed in curve order; a token that an
// earlier curve (or an earlier slot) already gave is dropped; the row is padded
// to k with -1.  Each curve's window follows the single-curve rule with k // curves
// in place of k.
//
// A warp owns 32 consecutive queries; each lane binary-searches its query in
// every curve's prefix, then the warp walks its 32 queries and, for each,
// gathers the curves' windows (one slot per lane and 32-slot block), drops
// repeats (match.any inside a block, broadcasts against earlier blocks) and
// compacts the survivors with ballots.
#include "common.cuh"

namespace zeta {
namespace {

constexpr int kMaxCurves = 8;

// KB blocks of 32 slots cover the k slots of a row.
template <typename K, int KB>
__global__ void select_curves_kernel(const K *__restrict__ qc, const K *__restrict__ pc,
                                     const int32_t *__restrict__ pidx, int32_t *__restrict__ out,
                                     int64_t S, int N, int C, int k, int64_t T, int curves) {
    const int64_t wpr = (N + 31) / 32;                    // warps per slice
    const int64_t gw = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    if (gw >= S * wpr) return;                            // whole warp exits together
    const int lane = threadIdx.x & 31;
    const unsigned lt = lanemask_lt();
    const int64_t seg = gw / wpr;
    const int qb = (int)(gw % wpr) * 32;
    const int i = qb + lane;
    const int km = k / curves;
    const int used = km * curves;                         // slots the windows fill
    int start[kMaxCurves];
#pragma unroll
    for (int m = 0; m < kMaxCurves; ++m) start[m] = -1;
    if (i < N) {
        const int c = i / C;
        if (c >= 1) {
            const int M = c * C;
#pragma unroll
            for (int m = 0; m < kMaxCurves; ++m) {
                if (m < curves) {
                    const K *p = pc + ((int64_t)m * S + seg) * T + (int64_t)C * c * (c - 1) / 2;
                    const K x = qc[((int64_t)m * S + seg) * N + i];
                    int lo = 0, hi = M;                    // upper bound
                    while (lo < hi) {
                        const int mid = (lo + hi) >> 1;
                        if (p[mid] <= x) lo = mid + 1; else hi = mid;
                    }
                    int s = lo - (km + 1) / 2;
                    s = s > M - km ? M - km : s;
                    start[m] = s < 0 ? 0 : s;
                }
            }
        }
    }
    const int last = min(32, N - qb);
    for (int qq = 0; qq < last; ++qq) {
        const int i2 = qb + qq;
        const int c2 = i2 / C;
        const int M2 = c2 * C;
        const int64_t off = (int64_t)C * c2 * (c2 - 1) / 2;
        int st[kMaxCurves];
#pragma unroll
        for (int m = 0; m < kMaxCurves; ++m) st[m] = __shfl_sync(kFull, start[m], qq);
        int e[KB];
#pragma unroll
        for (int b = 0; b < KB; ++b) {
            const int p = b * 32 + lane;
            int j = -1;
            if (c2 >= 1 && p < used) {
                const int m = p / km;
                const int u = p - m * km;
                int s = 0;
#pragma unroll
                for (int mm = 0; mm < kMaxCurves; ++mm) s = mm == m ? st[mm] : s;
                if (s + u < M2) j = __ldg(pidx + ((int64_t)m * S + seg) * T + off + s + u);
            }
            e[b] = j;
        }
        // A slot is a repeat when an earlier slot holds the same key.
        bool keep[KB];
#pragma unroll
        for (int b = 0; b < KB; ++b) {
            const unsigned same = __match_any_sync(kFull, e[b]);
            keep[b] = e[b] >= 0 && (same & lt) == 0;
        }
#pragma unroll
        for (int sb = 0; sb < KB - 1; ++sb) {
            if (sb * 32 >= used) break;                   // uniform across the warp
            for (int sl = 0; sl < 32; ++sl) {
                const int y = __shfl_sync(kFull, e[sb], sl);
#pragma unroll
                for (int b = sb + 1; b < KB; ++b) keep[b] = keep[b] && e[b] != y;
            }
        }
        int32_t *o = out + (seg * N + i2) * (int64_t)k;
        int cnt = 0;
#pragma unroll
        for (int b = 0; b < KB; ++b) {
            const unsigned bal = __ballot_sync(kFull, keep[b]);
            if (keep[b]) o[cnt + __popc(bal & lt)] = e[b];
            cnt += __popc(bal);
        }
        for (int t = cnt + lane; t < k; t += 32) o[t] = -1;
    }
}

template <typename K, int KB>
void launch_sel(const Prob &p, int curves, const void *q_codes, const void *prefix_codes,
                const int32_t *prefix_idx, int32_t *idx, cudaStream_t st) {
    const int64_t warps = p.S * ((p.N + 31) / 32);
    const int threads = 256;
    const int64_t blocks = (warps * 32 + threads - 1) / threads;
    select_curves_kernel<K, KB><<<(unsigned)blocks, threads, 0, st>>>(
        static_cast<const K *>(q_codes), static_cast<const K *>(prefix_codes), prefix_idx, idx,
        p.S, p.N, p.C, p.k, p.T, curves);
}

template <typename K>
void launch_sel_k(const Prob &p, int curves, const void *q_codes, const void *prefix_codes,
                  const int32_t *prefix_idx, int32_t *idx, cudaStream_t st) {
    const int kb = (p.k + 31) / 32;
    if (kb <= 1) launch_sel<K, 1>(p, curves, q_codes, prefix_codes, prefix_idx, idx, st);
    else if (kb <= 2) launch_sel<K, 2>(p, curves, q_codes, prefix_codes, prefix_idx, idx, st);
    else if (kb <= 4) launch_sel<K, 4>(p, curves, q_codes, prefix_codes, prefix_idx, idx, st);
    else launch_sel<K, 8>(p, curves, q_codes, prefix_codes, prefix_idx, idx, st);
}

}  // namespace

cudaError_t launch_select_curves(const Prob &p, int curves, const void *q_codes,
                                 const void *prefix_codes, const int32_t *prefix_idx,
                                 int32_t *idx, cudaStream_t st) {
    if (p.code64)
        launch_sel_k<uint64_t>(p, curves, q_codes, prefix_codes, prefix_idx, idx, st);
    else
        launch_sel_k<uint32_t>(p, curves, q_codes, prefix_codes, prefix_idx, idx, st);
    return cudaGetLastError();
}

}  // namespace zeta
