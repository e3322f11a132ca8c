// attend_fwd_tc.cuh -- fast forward for bf16 values with d_V = 64 and d_K <= 4
// (kernel template; attend_fwd_tc.cu launches it on a given selection,
// attend_fwd_fused.cu with the selection computed inside).
//
// Same definition as attend_fwd.cu (Cauchy softmax over window keys plus the
// own-chunk causal keys; OpenReview discussion of "ZETA: Leveraging Z-order
// Curves for Efficient Top-k Attention", reply A2 "Discussion on its
// robustness" and reply A3 "Justification for Euclidean Distance Claim"),
// organised for GB300:
//
//  * One CTA = 64 consecutive queries of one chunk (4 warps x 16 rows).
//  * Window part (a gather): a warp takes one query at a time; each lane owns
//    two selected keys (index, coordinates, Cauchy weight); the gathered
//    128-byte bf16 value rows come in with 32-byte loads (four lanes per row),
//    all 8 loads of a lane's 64-key pass in flight together, and the weighted
//    sum V^T w runs
//    on the tensor cores (rows transposed in registers by movmatrix, w in
//    column 0 of B); the next query's indices are fetched while the current
//    query is processed.  Partial sums (sum w v, sum w) go to shared memory in
//    float32.
//  * Own-chunk part (a dense causal C x C/2 x 64 contraction per chunk): key
//    tiles of 64 rows are staged by cp.async into XOR-swizzled shared memory
//    (double buffered); each thread builds its slice of the weight tile P
//    straight into mma A fragments (bf16), B fragments come from ldmatrix.trans,
//    and mma.sync m16n8k16 accumulates in float32 registers.  Row sums of P are
//    kept in float32 from the unrounded weights.
//  * The two partial sums simply add (Cauchy weights are in (0, 1], no
//    rescaling).  The other weight kernels (flags; reply A3 "Justification for
//    Euclidean Distance Claim") reuse everything: inverse Euclidean swaps the
//    weight; the softmax keeps a running shift (the smallest d2 seen) per query,
//    rescales its sums when the shift moves (per 64-key pass in the window, per
//    key tile in the own chunk, which starts from the window's shift) and
//    brings the window sums onto the final shift in the epilogue.
#pragma once

#include <type_traits>

#include "mma.cuh"

namespace zeta {
namespace {

constexpr int TQ = 64;            // queries per CTA
constexpr int TK = 64;            // keys per own-chunk tile
constexpr int DV = 64;
constexpr int THREADS = 128;
constexpr int WPAD = DV + 4;      // padded window-partial row

// Where the window indices come from.  NoSel: an idx array made by the select
// step.  FusedSel: the select step runs inside the kernel (each query's upper
// bound in its sorted prefix by binary search, the window is the contiguous
// run of the prefix's indices around it, OpenReview reply A3 "Chunking ..."),
// and the rows are written to idx_out for the backward.
struct NoSel {};
template <typename K>
struct FusedSel {
    using code_t = K;
    const K *qcodes;          // [S, N]
    const K *pcodes;          // [S, T]
    const int32_t *pidx;      // [S, T]
    int32_t *idx_out;         // [S, N, k]
    int64_t T;
};

// Column of window-partial dimension d: the eight lanes that store one query's
// sums write dimensions {0, 1, 16, 17, 32, 33, 48, 49} + 2 cb at once, which
// fall on four banks twice; flipping bit 1 in the upper half (d ^ 2 for
// d >= 32) spreads them over eight.  Adjacent even/odd dimensions stay adjacent.
__device__ __forceinline__ int wcol(int d) { return d ^ ((d >> 5) << 1); }

struct __align__(16) FwdSmem {
    __nv_bfloat16 v[2][TK * DV];  // swizzled: 16-byte chunk c of row r at c ^ (r & 7)
    float4 kt[2][TK];
    float win[TQ][WPAD];
    float swin[TQ];
    float mwin[TQ];               // softmax: the window's shift per query
};

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

// Stage own-chunk key tile `kt` (keys cC + kt*TK ...) into buffer b.
__device__ __forceinline__ void load_tile(FwdSmem &sm, int b, const float *kb,
                                          const __nv_bfloat16 *vb, int key0, int key_end,
                                          int dK) {
    const int t = threadIdx.x;
#pragma unroll
    for (int r = 0; r < (TK * DV / 8) / THREADS; ++r) {     // 4 chunks of 16 B per thread
        const int id = r * THREADS + t;
        const int row = id >> 3, ch = id & 7;
        const int key = key0 + row;
        const bool ok = key < key_end;
        const __nv_bfloat16 *src = vb + (int64_t)(ok ? key : key0) * DV + ch * 8;
        cp_async16(smem_u32(&sm.v[b][row * DV + ((ch ^ (row & 7)) * 8)]), src, ok ? 16 : 0);
    }
    if (t < TK) {
        const int key = key0 + t;
        float4 kk = make_float4(0.f, 0.f, 0.f, 0.f);
        if (key < key_end) {
            const float *p = kb + (int64_t)key * dK;
            kk.x = p[0];
            if (dK > 1) kk.y = p[1];
            if (dK > 2) kk.z = p[2];
            if (dK > 3) kk.w = p[3];
        }
        sm.kt[b][t] = kk;
    }
}

template <int DK, int WK, typename Sel>
__global__ void __launch_bounds__(THREADS, 4)
attend_fwd_tc(const float *__restrict__ q, const float *__restrict__ kx,
              const __nv_bfloat16 *__restrict__ v, const float *__restrict__ gamma,
              const int32_t *__restrict__ idx, __nv_bfloat16 *__restrict__ out,
              float *__restrict__ rowsum, int32_t *status, int N, int H, int k, int C,
              int tiles_per_chunk, Sel sel) {
    constexpr bool kFused = !std::is_same<Sel, NoSel>::value;
    __shared__ FwdSmem sm;
    const int64_t seg = blockIdx.y;
    const int c = blockIdx.x / tiles_per_chunk;
    const int qt = blockIdx.x % tiles_per_chunk;
    const int cC = c * C;
    const int cend = cC + C;
    const int i0 = cC + qt * TQ;
    const int iend = min(cend, i0 + TQ);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float gm = gamma[seg % H];
    const float inv_g2 = __frcp_rn(gm * gm);
    const float *kb = kx + seg * (int64_t)N * DK;
    const float *qb = q + seg * (int64_t)N * DK;
    const __nv_bfloat16 *vb = v + seg * (int64_t)N * DV;

    const int nkt = (iend - 1 - cC) / TK + 1;     // own-chunk key tiles up to the last query
    load_tile(sm, 0, kb, vb, cC, cend, DK);
    cp_async_commit();

    // ------------------------------------------------------ window part ---
    // A pass covers up to 64 selected keys: lane L owns slots L and L+32
    // (index, key coordinates, weight); the 16 value-row loads of the pass are
    // all issued before any is used, and the first pass's indices of the next
    // query are fetched while the current one is processed.  The weighted sum
    // runs on the tensor cores: for 16 selected keys, sum_j w_j v_j = V^T w is
    // four m16n8k16 mma (16 dimensions each) with w (bf16, like the own-chunk
    // P) in column 0 of B.  Lane (g, t) loads 16-byte slices 2t, 2t+1 of rows
    // g and g+8 of the 16 (one 32-byte access per row: each sector of a row is
    // requested once); movmatrix transposes them 8x8 block by block into
    // A fragments, and the sums stay in the mma's column-0 registers.
    const int wq0 = i0 + warp * 16;
    const int nqw = c > 0 ? max(0, min(16, iend - wq0)) : 0;
    const int g4 = lane >> 2, s4 = lane & 3;
    int wstart = 0;                 // fused: lane r < nqw holds query wq0 + r's window start
    if constexpr (kFused) {
        using K = typename Sel::code_t;
        if (c == 0) {               // chunk 0 selects nothing
            const int nr = max(0, min(16, iend - wq0));
            for (int r = 0; r < nr; ++r)
                for (int t = lane; t < k; t += 32) sel.idx_out[(seg * N + wq0 + r) * (int64_t)k + t] = -1;
        } else {
            // Upper bound of each query's code in its prefix (the number of keys
            // with code <= the query's), in two levels: the first code of every
            // block of 2^fsh prefix entries (a fence) is staged in shared memory
            // (the window partials' space, unused until the first query is done)
            // and searched there; the query's block is then searched in global
            // memory, where its probes after the first hit L1.  Same result as
            // one binary search over the prefix, with far fewer dependent loads
            // from L2 before the first gather.
            const K *pc = sel.pcodes + seg * sel.T + (int64_t)C * c * (c - 1) / 2;
            K *fence = reinterpret_cast<K *>(&sm.win[0][0]);
            constexpr int kFenceMax = (int)(sizeof(sm.win) / sizeof(K));
            int fsh = 6;
            while ((cC >> fsh) >= kFenceMax) ++fsh;
            const int nf = (cC + (1 << fsh) - 1) >> fsh;
            for (int f = threadIdx.x; f < nf; f += THREADS) fence[f] = pc[(int64_t)f << fsh];
            __syncthreads();
            if (lane < nqw) {
                const K x = sel.qcodes[seg * N + wq0 + lane];
                int lo = 0, hi = nf;           // fences with code <= x
                while (lo < hi) {
                    const int mid = (lo + hi) >> 1;
                    if (fence[mid] <= x) lo = mid + 1; else hi = mid;
                }
                int r = 0;
                if (lo > 0) {                  // entry b0 (the fence) is <= x; later blocks are > x
                    const int b0 = (lo - 1) << fsh;
                    int a = b0 + 1, b = min(cC, b0 + (1 << fsh));
                    while (a < b) {
                        const int mid = (a + b) >> 1;
                        if (pc[mid] <= x) a = mid + 1; else b = mid;
                    }
                    r = a;
                }
                int s0 = r - (k + 1) / 2;
                s0 = s0 > cC - k ? cC - k : s0;
                wstart = s0 < 0 ? 0 : s0;
            }
            __syncthreads();                   // fences read before any window partial is written
        }
    }
    auto load_idx = [&](int i, int t0, int (&j)[2]) {
        if constexpr (kFused) {
            const int st = __shfl_sync(kFull, wstart, i - wq0);
            const int32_t *src = sel.pidx + seg * sel.T + (int64_t)C * c * (c - 1) / 2 + st + t0;
            int32_t *dst = sel.idx_out + (seg * N + i) * (int64_t)k + t0;
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                const int t = t0 + s * 32 + lane;
                j[s] = t < k ? __ldg(src + s * 32 + lane) : -1;
                if (t < k) dst[s * 32 + lane] = j[s];
            }
        } else {
            const int32_t *irow = idx + (seg * N + i) * (int64_t)k + t0;
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                const int t = t0 + s * 32 + lane;
                j[s] = t < k ? __ldg(irow + s * 32 + lane) : -1;
            }
        }
    };
    int jn[2] = {-1, -1};
    if (nqw > 0) load_idx(wq0, 0, jn);
    for (int r = 0; r < 16; ++r) {
        const int row = warp * 16 + r;
        float cacc[4][4];           // column 0 of four 16-dimension mma tiles
#pragma unroll
        for (int cb = 0; cb < 4; ++cb)
#pragma unroll
            for (int e = 0; e < 4; ++e) cacc[cb][e] = 0.f;
        float sw = 0.f;
        float mrun = INFINITY;                     // softmax shift of this query
        if (r < nqw) {
            const int i = wq0 + r;
            float qi[4];
#pragma unroll
            for (int d = 0; d < 4; ++d) qi[d] = d < DK ? qb[(int64_t)i * DK + d] : 0.f;
            for (int t0 = 0; t0 < k; t0 += 64) {
                int j[2] = {jn[0], jn[1]};
                if (t0 + 64 < k) {
                    load_idx(i, t0 + 64, jn);              // next pass of this query
                } else if (r + 1 < nqw) {
                    load_idx(i + 1, 0, jn);                // first pass of the next query
                }
                float4 kk[2];
#pragma unroll
                for (int s = 0; s < 2; ++s) {
                    if (j[s] != -1 && (unsigned)j[s] >= (unsigned)cC) {
                        set_status(status, ZETA_ERR_BOUNDS);
                        j[s] = -1;
                    }
                    kk[s] = j[s] >= 0 ? load_k4(kb + (int64_t)j[s] * DK, DK)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
                }
                const int nmt = min(4, (k - t0 + 15) >> 4);  // 16-key tiles in this pass
                uint4 buf[4][4];                    // rows g, g+8 of tile mt: slices 2t, 2t+1
#pragma unroll
                for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int slot = 16 * mt + 8 * h + g4;
                        const int jr = __shfl_sync(kFull, j[mt >> 1], slot & 31);
                        const bool ok = mt < nmt && jr >= 0;
                        ld_stream32(vb + (int64_t)(ok ? jr : 0) * DV + s4 * 16, ok, buf[mt][2 * h],
                                    buf[mt][2 * h + 1]);
                    }
                }
                float d2v[2];
#pragma unroll
                for (int s = 0; s < 2; ++s) d2v[s] = j[s] >= 0 ? dist2k<DK>(qi, kk[s]) : INFINITY;
                if constexpr (WK == kWSoftmax) {
                    float pm = fminf(d2v[0], d2v[1]);
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) pm = fminf(pm, __shfl_xor_sync(kFull, pm, o));
                    const float mn = fminf(mrun, pm);
                    if (mn != mrun) {                    // uniform across the warp
                        const float sc = shift_scale(mn, mrun, inv_g2);
#pragma unroll
                        for (int cb = 0; cb < 4; ++cb)
#pragma unroll
                            for (int e = 0; e < 4; ++e) cacc[cb][e] *= sc;
                        sw *= sc;
                        mrun = mn;
                    }
                }
                float w[2];
#pragma unroll
                for (int s = 0; s < 2; ++s) {
                    w[s] = j[s] >= 0 ? weight_fast<WK>(d2v[s], mrun, inv_g2) : 0.f;
                    sw += w[s];
                }
#pragma unroll
                for (int mt = 0; mt < 4; ++mt) {
                    if (mt < nmt) {
                        // weights of slots 16mt + 2t, +1, +8, +9 (owner lane = slot % 32)
                        const int sb = 16 * mt + 2 * s4;
                        const float e0 = __shfl_sync(kFull, w[mt >> 1], sb & 31);
                        const float e1 = __shfl_sync(kFull, w[mt >> 1], (sb + 1) & 31);
                        const float e2 = __shfl_sync(kFull, w[mt >> 1], (sb + 8) & 31);
                        const float e3 = __shfl_sync(kFull, w[mt >> 1], (sb + 9) & 31);
                        const uint32_t ba = g4 == 0 ? pack_bf16(e0, e1) : 0u;
                        const uint32_t bb = g4 == 0 ? pack_bf16(e2, e3) : 0u;
                        const uint32_t ra0[4] = {buf[mt][0].x, buf[mt][0].y, buf[mt][0].z, buf[mt][0].w};
                        const uint32_t ra1[4] = {buf[mt][1].x, buf[mt][1].y, buf[mt][1].z, buf[mt][1].w};
                        const uint32_t rb0[4] = {buf[mt][2].x, buf[mt][2].y, buf[mt][2].z, buf[mt][2].w};
                        const uint32_t rb1[4] = {buf[mt][3].x, buf[mt][3].y, buf[mt][3].z, buf[mt][3].w};
#pragma unroll
                        for (int cb = 0; cb < 4; ++cb) {   // dims 16 (m/2) + 8 h + 2 cb + (m%2)
                            const uint32_t af[4] = {movmatrix_trans(ra0[cb]), movmatrix_trans(ra1[cb]),
                                                    movmatrix_trans(rb0[cb]), movmatrix_trans(rb1[cb])};
                            mma16816(cacc[cb], af, ba, bb);
                        }
                    }
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sw += __shfl_xor_sync(kFull, sw, o);
        }
        if (s4 == 0) {              // lane 4m holds mma rows m and m+8 of column 0
            const int d0 = 16 * (g4 >> 1) + (g4 & 1);
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) {
                sm.win[row][wcol(d0 + 2 * cb)] = cacc[cb][0];
                sm.win[row][wcol(d0 + 8 + 2 * cb)] = cacc[cb][2];
            }
        }
        if (lane == 0) {
            sm.swin[row] = sw;
            sm.mwin[row] = mrun;
        }
    }
    __syncwarp();

    // --------------------------------------------------- own-chunk part ---
    const int g = lane >> 2, tig = lane & 3;
    const int ra = i0 + warp * 16 + g, rb = ra + 8;
    float qa[4], qbv[4];
#pragma unroll
    for (int d = 0; d < 4; ++d) {
        qa[d] = (ra < iend && d < DK) ? qb[(int64_t)ra * DK + d] : 0.f;
        qbv[d] = (rb < iend && d < DK) ? qb[(int64_t)rb * DK + d] : 0.f;
    }
    const int lim_a = ra < iend ? ra : -1;        // last key index row a may see
    const int lim_b = rb < iend ? rb : -1;
    float2 qab[4];                                // (row a, row b) coordinates
#pragma unroll
    for (int d = 0; d < 4; ++d) qab[d] = make_float2(qa[d], qbv[d]);
    const float2 ig2 = dup2(inv_g2);
    const int rowa = warp * 16 + g, rowb = rowa + 8;
    float2 mab = make_float2(sm.mwin[rowa], sm.mwin[rowb]);   // softmax shifts of rows a, b
    float acc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
    float2 sab = make_float2(0.f, 0.f);           // row sums of rows a, b
    const int warp_first = i0 + warp * 16;
    const int warp_last = min(warp_first + 15, iend - 1);
    const bool warp_rows_full = warp_first + 15 < iend;

    // Squared distances of rows (a, b) to key kl of the tile.
    auto d2ab = [&](const float4 *Ks, int kl) {
        const float4 kv = Ks[kl];
        const float kc[4] = {kv.x, kv.y, kv.z, kv.w};
        float2 d2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int d = 0; d < DK; ++d) {
            const float2 e = sub2(qab[d], dup2(kc[d]));
            d2 = fma2(e, e, d2);
        }
        return d2;
    };

    // One 64-key tile: weights of rows (a, b) against 16 keys per k-step, packed.
    auto tile = [&](const float4 *Ks, uint32_t vbase, int key0, auto masked) {
        if constexpr (WK == kWSoftmax) {           // move the shift to this tile's minimum
            float2 tmin = make_float2(INFINITY, INFINITY);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const int kl = ks * 16 + 2 * tig + (h & 1) + (h >> 1) * 8;
                    float2 d2 = d2ab(Ks, kl);
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
            const float sa_ = shift_scale(mn.x, mab.x, inv_g2);
            const float sb_ = shift_scale(mn.y, mab.y, inv_g2);
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                acc[nt][0] *= sa_;
                acc[nt][1] *= sa_;
                acc[nt][2] *= sb_;
                acc[nt][3] *= sb_;
            }
            sab = mul2(sab, make_float2(sa_, sb_));
            mab = mn;
        }
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            const int kk0 = ks * 16 + 2 * tig;
            float wv[8];
#pragma unroll
            for (int h = 0; h < 4; ++h) {              // keys kk0, kk0+1, kk0+8, kk0+9
                const int kl = kk0 + (h & 1) + (h >> 1) * 8;
                float2 w = weight_fast2<WK>(d2ab(Ks, kl), mab, ig2);
                if (decltype(masked)::value) {
                    const int key = key0 + kl;
                    w.x = key <= lim_a ? w.x : 0.f;
                    w.y = key <= lim_b ? w.y : 0.f;
                }
                wv[h] = w.x;
                wv[4 + h] = w.y;
                sab = add2(sab, w);
            }
            uint32_t a[4];
            a[0] = pack_bf16(wv[0], wv[1]);
            a[1] = pack_bf16(wv[4], wv[5]);
            a[2] = pack_bf16(wv[2], wv[3]);
            a[3] = pack_bf16(wv[6], wv[7]);
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                const int m = lane >> 3, rr = lane & 7;
                const int key = ks * 16 + (m & 1) * 8 + rr;
                uint32_t b[4];
                ldsm_x4_trans(b, vbase + (uint32_t)swz(key, np * 2 + (m >> 1)) * 2u);
                mma16816(acc[2 * np], a, b[0], b[1]);
                mma16816(acc[2 * np + 1], a, b[2], b[3]);
            }
        }
    };

    for (int kt = 0; kt < nkt; ++kt) {
        if (kt + 1 < nkt) load_tile(sm, (kt + 1) & 1, kb, vb, cC + (kt + 1) * TK, cend, DK);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        const int key0 = cC + kt * TK;
        if (key0 <= warp_last) {                   // else every weight of this warp is 0
            const float4 *Ks = sm.kt[kt & 1];
            const uint32_t vbase = smem_u32(sm.v[kt & 1]);
            if (warp_rows_full && key0 + TK - 1 <= warp_first)
                tile(Ks, vbase, key0, std::false_type{});
            else
                tile(Ks, vbase, key0, std::true_type{});
        }
        __syncthreads();
    }
    float sa = sab.x, sb = sab.y;

    // --------------------------------------------------------- epilogue ---
    sa += __shfl_xor_sync(kFull, sa, 1);
    sa += __shfl_xor_sync(kFull, sa, 2);
    sb += __shfl_xor_sync(kFull, sb, 1);
    sb += __shfl_xor_sync(kFull, sb, 2);
    // Window sums onto the final shift (softmax; a factor of 1 otherwise).
    float fa = 1.f, fb = 1.f;
    if constexpr (WK == kWSoftmax) {
        fa = shift_scale(mab.x, sm.mwin[rowa], inv_g2);
        fb = shift_scale(mab.y, sm.mwin[rowb], inv_g2);
    }
    const float ta = sa + sm.swin[rowa] * fa, tb = sb + sm.swin[rowb] * fb;
    const float ia = ra < iend ? __frcp_rn(ta) : 0.f;
    const float ib = rb < iend ? __frcp_rn(tb) : 0.f;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
        const int col = nt * 8 + 2 * tig;
        if (ra < iend) {
            const float o0 = __fmaf_rn(sm.win[rowa][wcol(col)], fa, acc[nt][0]) * ia;
            const float o1 = __fmaf_rn(sm.win[rowa][wcol(col) + 1], fa, acc[nt][1]) * ia;
            *reinterpret_cast<__nv_bfloat162 *>(out + (seg * N + ra) * (int64_t)DV + col) =
                __floats2bfloat162_rn(o0, o1);
        }
        if (rb < iend) {
            const float o0 = __fmaf_rn(sm.win[rowb][wcol(col)], fb, acc[nt][2]) * ib;
            const float o1 = __fmaf_rn(sm.win[rowb][wcol(col) + 1], fb, acc[nt][3]) * ib;
            *reinterpret_cast<__nv_bfloat162 *>(out + (seg * N + rb) * (int64_t)DV + col) =
                __floats2bfloat162_rn(o0, o1);
        }
    }
    if (tig == 0) {
        if (ra < iend) rowsum[seg * N + ra] = ta;
        if (rb < iend) rowsum[seg * N + rb] = tb;
    }
}

}  // namespace
}  // namespace zeta
