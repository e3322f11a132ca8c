// bwd_own_tc05.cu -- the key side of the backward's own-chunk block on the
// Blackwell tensor cores (tcgen05 + TMEM, TMA-fed).
//
// Passages: "ZETA: Leveraging Z-order Curves for Efficient Top-k Attention",
// the chunked causal selection (a query scores the keys of its own chunk up to
// itself exactly), and the Cauchy weights w = 1 / (1 + d^2 / gamma^2) (the
// other weight kernels of reply A3 "Justification for Euclidean Distance
// Claim" swap in their w and dw/d(d^2)); gradients with the selection held
// fixed.  For key j of chunk c and the queries i >= j of the same chunk:
//   g_ij = dO_i . v_j,   a_ij = w_ij / s_i,
//   dv_j += sum_i a_ij dO_i,
//   dk_j += sum_i (g_ij - gbar_i) / s_i * (-dw/d(d^2))_ij * 2 (q_i - k_j)
// (the Cauchy constant 2 / gamma^2 of -dw/d(d^2) = w^2 / gamma^2 is applied
// where the partial sums are combined).  s_i, gbar_i (and the softmax shift)
// come from the query side's per-query records.
//
// Unit: 128 keys of one chunk (the accumulators' 128 TMEM lanes) against the
// chunk's query tiles of 128 from the key tile on.  Per query tile:
//   GEMM1  G^T = V_keys . dO_tile^T   M = 128 keys, N = 128 queries, K = 64
//   element-wise: a thread owns one key row and a quarter of the tile's
//          queries; it reads its 32 values of G^T (tcgen05.ld), forms w, a and
//          the dk terms (summed in registers) and writes a as bf16 into P^T, a
//          K-major tile with the 128-byte swizzle (two 64-query K blocks)
//   GEMM2  dV += P^T . dO_tile       M = 128 keys, N = 64, K = 128 queries;
//          dO_tile is the MN-major B operand (the same swizzled tile as in
//          GEMM1, where it is the K-major B)
// The kernel is persistent and warp-specialised:
//   warp 0     producer: the unit's value tile and each query tile's dO rows
//              by TMA, the unit's key coordinates by bulk copy, the tile's
//              query records transposed into shared memory (one array per
//              field) by the warp's lanes;
//   warp 1     MMA issuer (one thread) and owner of the TMEM allocation: two
//              128-column G^T buffers and two 64-column dV accumulators (the
//              units alternate); one stream of tiles across units, GEMM1 of a
//              tile issued before GEMM2 of the tile before it;
//   warps 2-17 element-wise, four warps per TMEM lane quarter (a warp may
//              only read the lane quarter of its index mod 4); a unit's
//              epilogue (its dV rows from TMEM, the dk sums) runs after the
//              next unit's first tile, when that unit's last GEMM2 is done.
// The units of a chunk are handed out in pairs (key tiles p and n-1-p: the same
// number of query tiles per pair) to neighbouring CTAs, so that the chunk's dO
// rows are read from L2.  Output per key: dv (64 floats) and dk (4 floats, the
// four query parts' sums added through shared memory, handed over by
// mbarriers), partial sums that the key walk's epilogue adds to its own.  No
// wait is on a hardware barrier among the element-wise warps, so that a warp
// that gives up cannot leave the others blocked.
// Hand-offs are mbarriers; every wait is bounded; a wait that gives up records
// ZETA_ERR_DEVICE_TIMEOUT and raises an abort flag that ends every role's loop,
// after which the producer waits (bounded) for its copies in flight and the MMA
// thread for its MMAs before the TMEM is freed.
#include <type_traits>

#include "bwd_rec.cuh"
#include "f2x.cuh"
#include "tc05.cuh"
#include "tmap.cuh"

namespace zeta {
namespace {

constexpr int OKR = 128;                  // keys per unit
constexpr int OQ = 128;                   // queries per tile
constexpr int ODV = 64;                   // d_V
constexpr int OSTG = 5;                   // dO stages
constexpr int OEPI = 16;                  // element-wise warps (OEPI / 4 per TMEM lane quarter)
constexpr int OPARTS = OEPI / 4;          // query parts of a tile
constexpr int OPART = OQ / OPARTS;        // queries of a tile per element-wise warp
constexpr int OCH = OPART / 8;            // 8-query chunks per warp and tile
// producer, MMA, element-wise warps, and two spare warps that only take part in
// the set-up and the final barrier: registers are granted per four warps, so a
// block of 18 warps gets no more per thread than one of 20
constexpr int OSPARE = OEPI == 16 ? 2 : 0;
constexpr int OTHREADS = 64 + 32 * OEPI + 32 * OSPARE;
constexpr uint32_t V_BYTES = OKR * ODV * 2;
constexpr uint32_t D_BYTES = OQ * ODV * 2;
constexpr uint32_t P_BLOCK = OKR * 64 * 2;     // one 64-query K block of P^T
constexpr uint32_t P_BYTES = 2 * P_BLOCK;
constexpr uint32_t TM_DV = 2 * OQ;              // TMEM columns: G^T x 2, then dV x 2
constexpr uint32_t TM_COLS = 512;
constexpr int kRecFields = 8;                   // q0..q3, 1/s, -gbar/s, m, unused

struct OwnRecs {
    float f[kRecFields][OQ];
};

struct OwnHead {
    uint64_t v_full[2], v_empty[2];
    uint64_t d_full[OSTG], d_empty[OSTG];
    uint64_t g_full[2], g_empty[2];
    uint64_t p_full[2], p_empty[2];
    uint64_t dv_full[2], dv_empty[2];
    uint64_t red_full[2], red_free[2];    // a unit's dk parts written / read
    uint64_t drain;
    uint32_t tmem_base;
    int32_t abort;
};

constexpr uint32_t OFF_V = 0;
constexpr uint32_t OFF_D = OFF_V + 2 * V_BYTES;
constexpr uint32_t OFF_P = OFF_D + OSTG * D_BYTES;
constexpr uint32_t OFF_R = OFF_P + 2 * P_BYTES;
constexpr uint32_t OFF_K = OFF_R + OSTG * sizeof(OwnRecs);     // dk parts [2][parts][128] float4
constexpr uint32_t OFF_KC = OFF_K + 2 * OPARTS * OKR * 16;      // key coordinates [2][128 * 4]
constexpr int kMaxHeads = 64;                                   // gammas staged in shared memory
constexpr uint32_t OFF_G = OFF_KC + 2 * OKR * 16;
constexpr uint32_t OFF_H = OFF_G + kMaxHeads * 4;
constexpr size_t kOwnSmem = 1024 + OFF_H + sizeof(OwnHead);

__device__ __forceinline__ bool own_aborted(const OwnHead &sh) {
    return *reinterpret_cast<const volatile int32_t *>(&sh.abort) != 0;
}

__device__ __forceinline__ bool own_wait(OwnHead &sh, uint64_t *bar, uint32_t parity,
                                         int32_t *status) {
    if (mbar_wait_bounded(bar, parity)) return true;
    *reinterpret_cast<volatile int32_t *>(&sh.abort) = 1;
    set_status(status, ZETA_ERR_DEVICE_TIMEOUT);
    return false;
}

// Unit u (a key tile) of the pair order: chunk u / nkt, then key tiles
// 0, nkt-1, 1, nkt-2, ...
struct OwnUnit {
    int64_t seg;
    int c, kt;
};
__device__ __forceinline__ OwnUnit own_unit(int64_t u, int nch, int nkt) {
    const int64_t sc = u / nkt;
    const int r = (int)(u - sc * nkt);
    OwnUnit o;
    o.seg = sc / nch;
    o.c = (int)(sc - o.seg * nch);
    o.kt = (r & 1) ? nkt - 1 - (r >> 1) : (r >> 1);
    return o;
}

// Raise the barrier's expected transaction count without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

template <int DK, int WK>
__global__ void __launch_bounds__(OTHREADS, 1)
bwd_key_own_tc05(const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap dmap,
                 const float *__restrict__ kx, const float *__restrict__ gamma,
                 const QRec *__restrict__ rec, float *__restrict__ own_dv,
                 float *__restrict__ own_dk, int N, int H, int C, int64_t units,
                 int32_t *status) {
    extern __shared__ unsigned char dsm[];
    unsigned char *base = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(dsm) + 1023) & ~uintptr_t(1023));
    OwnHead &sh = *reinterpret_cast<OwnHead *>(base + OFF_H);
    OwnRecs *recs = reinterpret_cast<OwnRecs *>(base + OFF_R);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nch = N / C, nkt = C / OKR;

    float *gsm = reinterpret_cast<float *>(base + OFF_G);
    for (int h = tid; h < H; h += blockDim.x) gsm[h] = gamma[h];
    if (tid == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sh.v_full[b], 1);
            mbar_init(&sh.v_empty[b], 1 + OEPI);   // last GEMM1 of the unit + key coordinates read
            mbar_init(&sh.g_full[b], 1);
            mbar_init(&sh.g_empty[b], OEPI);
            mbar_init(&sh.p_full[b], OEPI);
            mbar_init(&sh.p_empty[b], 1);
        }
        for (int s = 0; s < OSTG; ++s) {
            mbar_init(&sh.d_full[s], 32);        // every producer lane (records), + TMA bytes
            mbar_init(&sh.d_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sh.dv_full[b], 1);
            mbar_init(&sh.dv_empty[b], OEPI);
            mbar_init(&sh.red_full[b], OEPI);    // every element-wise warp's parts
            mbar_init(&sh.red_free[b], 4);       // read by the four part-0 warps
        }
        mbar_init(&sh.drain, 1);
        sh.abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&sh.tmem_base, TM_COLS);
        tmem_relinquish();
    }
    tc05_fence_before();
    __syncthreads();
    tc05_fence_after();
    const uint32_t tmem = sh.tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------ producer ---
        uint32_t v_iss[2] = {0u, 0u}, d_iss[OSTG] = {};
        uint32_t T = 0, U = 0;
        bool ok = true;
        for (int64_t pr = blockIdx.x; 2 * pr < units && ok; pr += gridDim.x) {
            for (int64_t u = 2 * pr; u < 2 * pr + 2 && u < units && ok; ++u, ++U) {
                if (__any_sync(kFull, own_aborted(sh))) { ok = false; break; }
                const OwnUnit w = own_unit(u, nch, nkt);
                const int j0 = w.c * C + w.kt * OKR;
                const int64_t row0 = w.seg * (int64_t)N;
                const uint32_t vb = U & 1u;
                if (lane == 0) {
                    ok = own_wait(sh, &sh.v_empty[vb], ((U >> 1) & 1u) ^ 1u, status);
                    if (ok) {
                        // the value tile and the unit's key coordinates (128 DK floats)
                        mbar_arrive_expect_tx(&sh.v_full[vb], V_BYTES + OKR * DK * 4);
                        tma_load_2d(base + OFF_V + vb * V_BYTES, &vmap, 0, (int)(row0 + j0),
                                    &sh.v_full[vb]);
                        bulk_load(base + OFF_KC + vb * (OKR * 16), kx + (row0 + j0) * DK, OKR * DK * 4,
                                  &sh.v_full[vb]);
                        ++v_iss[vb];
                    }
                }
                ok = __shfl_sync(kFull, ok, 0);
                const int ntile = nkt - w.kt;
                for (int t = 0; t < ntile && ok; ++t, ++T) {
                    const uint32_t s = T % OSTG;
                    if (lane == 0) ok = own_wait(sh, &sh.d_empty[s], ((T / OSTG) & 1u) ^ 1u, status);
                    ok = __shfl_sync(kFull, ok, 0);
                    if (!ok) break;
                    const int i0 = j0 + t * OQ;
                    if (lane == 0) {             // the dO rows first: their copy overlaps the records'
                        mbar_expect_tx(&sh.d_full[s], D_BYTES);
                        tma_load_2d(base + OFF_D + s * D_BYTES, &dmap, 0, (int)(row0 + i0),
                                    &sh.d_full[s]);
                        ++d_iss[s];
                    }
                    OwnRecs &rs = recs[s];
#pragma unroll
                    for (int x = 0; x < OQ / 32; ++x) {
                        const int ql = x * 32 + lane;
                        const float4 *src = reinterpret_cast<const float4 *>(rec + row0 + i0 + ql);
                        const float4 a = __ldg(src), b = __ldg(src + 1);
                        rs.f[0][ql] = a.x;
                        rs.f[1][ql] = a.y;
                        rs.f[2][ql] = a.z;
                        rs.f[3][ql] = a.w;
                        rs.f[4][ql] = b.x;
                        rs.f[5][ql] = b.y;
                        rs.f[6][ql] = b.z;
                    }
                    mbar_arrive(&sh.d_full[s]);  // each lane once its records are stored
                }
            }
        }
        if (lane == 0 && own_aborted(sh)) {
            // the last copy into each buffer completes after all earlier ones
            for (int b = 0; b < 2; ++b)
                if (v_iss[b]) mbar_wait_bounded(&sh.v_full[b], (v_iss[b] - 1u) & 1u);
            for (int s = 0; s < OSTG; ++s)
                if (d_iss[s]) mbar_wait_bounded(&sh.d_full[s], (d_iss[s] - 1u) & 1u);
        }
    } else if (warp == 1) {
        // --------------------------------------------------------- MMA ---
        if (lane == 0) {
            constexpr uint32_t idesc1 = idesc_bf16_f32(OKR, OQ);
            constexpr uint32_t idesc2 = idesc_bf16_f32(OKR, ODV) | (1u << 16);   // B MN-major
            const uint32_t sV = smem_u32(base + OFF_V), sD = smem_u32(base + OFF_D);
            const uint32_t sP = smem_u32(base + OFF_P);
            uint32_t T = 0, U = 0;
            bool issued = false, ok = true;
            // One stream of tiles across the units: GEMM1 of a tile, then GEMM2
            // of the tile before it (whatever unit that was), so that the first
            // G^T of a unit is ready when the element-wise warps finish the last
            // tile of the previous one.  A unit's dV goes to accumulator U & 1.
            struct Pend {
                uint32_t Tt, U;
                int tt;
                bool last, valid;
            } pend = {0u, 0u, 0, false, false};
            auto gemm2 = [&](const Pend &q) -> bool {      // dV (+)= P^T . dO of tile q
                const uint32_t b = q.Tt & 1u, s = q.Tt % OSTG, a = q.U & 1u;
                if (q.tt == 0 && !own_wait(sh, &sh.dv_empty[a], ((q.U >> 1) & 1u) ^ 1u, status))
                    return false;
                if (!own_wait(sh, &sh.p_full[b], (q.Tt >> 1) & 1u, status)) return false;
                tc05_fence_after();
                const uint32_t pa = sP + b * P_BYTES, db = sD + s * D_BYTES;
#pragma unroll
                for (int kk = 0; kk < OQ / 16; ++kk) {
                    const uint64_t ad = sdesc_k128(pa + (uint32_t)(kk >> 2) * P_BLOCK) + 2u * (kk & 3);
                    const uint64_t bd = sdesc_k128(db) + 128u * kk;   // 16 rows = 2048 bytes
                    umma_bf16(tmem + TM_DV + a * ODV, ad, bd, idesc2, (q.tt | kk) != 0);
                }
                umma_commit(&sh.p_empty[b]);
                umma_commit(&sh.d_empty[s]);
                if (q.last) umma_commit(&sh.dv_full[a]);
                return true;
            };
            for (int64_t pr = blockIdx.x; 2 * pr < units && ok; pr += gridDim.x) {
                for (int64_t u = 2 * pr; u < 2 * pr + 2 && u < units && ok; ++u, ++U) {
                    if (own_aborted(sh)) { ok = false; break; }
                    const OwnUnit w = own_unit(u, nch, nkt);
                    const int ntile = nkt - w.kt;
                    const uint32_t vb = U & 1u;
                    if (!(ok = own_wait(sh, &sh.v_full[vb], (U >> 1) & 1u, status))) break;
                    for (int t = 0; t < ntile; ++t) {
                        const uint32_t Tt = T + t, s = Tt % OSTG, b = Tt & 1u;
                        if (!(ok = own_wait(sh, &sh.d_full[s], (Tt / OSTG) & 1u, status))) break;
                        if (!(ok = own_wait(sh, &sh.g_empty[b], ((Tt >> 1) & 1u) ^ 1u, status))) break;
                        tc05_fence_after();
                        const uint64_t ad = sdesc_k128(sV + vb * V_BYTES);
                        const uint64_t bd = sdesc_k128(sD + s * D_BYTES);
#pragma unroll
                        for (int kk = 0; kk < ODV / 16; ++kk)
                            umma_bf16(tmem + b * OQ, ad + 2u * kk, bd + 2u * kk, idesc1, kk != 0);
                        issued = true;
                        umma_commit(&sh.g_full[b]);
                        if (t == ntile - 1) umma_commit(&sh.v_empty[vb]);
                        if (pend.valid && !(ok = gemm2(pend))) break;
                        pend = {Tt, U, t, t == ntile - 1, true};
                    }
                    if (!ok) break;
                    T += ntile;
                }
            }
            if (ok && pend.valid) ok = gemm2(pend);
            if (issued && own_aborted(sh)) {
                umma_commit(&sh.drain);
                mbar_wait_bounded(&sh.drain, 0);
            }
        }
    } else if (warp < 2 + OEPI) {
        // -------------------------------------------------- element-wise ---
        const int quarter = warp & 3;                    // TMEM lanes 32 quarter ..
        const int part = (warp - 2) >> 2;                // queries 32 part .. of each tile
        const int row = quarter * 32 + lane;             // key row of the unit
        const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
        // this thread's row of P^T in the K block of its queries
        const uint32_t sP = smem_u32(base + OFF_P) + (uint32_t)(row >> 3) * 1024u +
                            (uint32_t)(row & 7) * 128u;
        float4 *red = reinterpret_cast<float4 *>(base + OFF_K);     // [buffer][part][row]
        const uint32_t sR = smem_u32(base + OFF_R);                  // the stages' records
        uint32_t T = 0, U = 0;
        bool ok = true;
        // The epilogue of a unit (its dV row from TMEM, the dk parts summed
        // through shared memory) runs after the first tile of the next unit,
        // by which time the unit's last GEMM2 has long completed.
        bool pend = false;
        uint32_t pU = 0;
        int64_t pgj = 0;
        auto epilogue = [&]() -> bool {
            const uint32_t a = pU & 1u;
            bool okw = own_wait(sh, &sh.dv_full[a], (pU >> 1) & 1u, status);
            if (!__all_sync(kFull, okw)) return false;
            tc05_fence_after();
            constexpr int DVC = ODV / OPARTS;            // dV columns per warp
            uint32_t dr[DVC];
            if constexpr (DVC == 16)
                tmem_ld16(tl + TM_DV + a * ODV + DVC * part, *reinterpret_cast<uint32_t(*)[16]>(dr));
            else
                tmem_ld32(tl + TM_DV + a * ODV + DVC * part, *reinterpret_cast<uint32_t(*)[32]>(dr));
            tmem_ld_wait();
            tc05_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.dv_empty[a]);
            float4 *dst = reinterpret_cast<float4 *>(own_dv + pgj * ODV + DVC * part);
#pragma unroll
            for (int x = 0; x < DVC / 4; ++x)
                dst[x] = make_float4(__uint_as_float(dr[4 * x]), __uint_as_float(dr[4 * x + 1]),
                                     __uint_as_float(dr[4 * x + 2]), __uint_as_float(dr[4 * x + 3]));
            if (part == 0) {                             // the unit's dk: its parts summed
                okw = own_wait(sh, &sh.red_full[a], (pU >> 1) & 1u, status);
                if (!__all_sync(kFull, okw)) return false;
                const float4 *rb = red + a * (OPARTS * OKR);
                float4 s4 = rb[row];
#pragma unroll
                for (int x = 1; x < OPARTS; ++x) {
                    const float4 b2 = rb[x * OKR + row];
                    s4 = make_float4(s4.x + b2.x, s4.y + b2.y, s4.z + b2.z, s4.w + b2.w);
                }
                *reinterpret_cast<float4 *>(own_dk + pgj * 4) = s4;
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.red_free[a]);
            }
            return true;
        };
        for (int64_t pr = blockIdx.x; 2 * pr < units && ok; pr += gridDim.x) {
            for (int64_t u = 2 * pr; u < 2 * pr + 2 && u < units && ok; ++u, ++U) {
                if (__any_sync(kFull, own_aborted(sh))) { ok = false; break; }
                const OwnUnit w = own_unit(u, nch, nkt);
                const int ntile = nkt - w.kt;
                const int j = w.c * C + w.kt * OKR + row;
                const int64_t gj = w.seg * (int64_t)N + j;
                const float g0 = gsm[w.seg % H];
                // the unit's key coordinates arrive with its value tile
                bool okv = own_wait(sh, &sh.v_full[U & 1u], (U >> 1) & 1u, status);
                if (!__all_sync(kFull, okv)) { ok = false; break; }
                const float ig2s = __frcp_rn(g0 * g0);
                const F2 ig2 = f2_dup(ig2s), two_ig2 = f2_dup(2.f * ig2s), one2 = f2_dup(1.f);
                const float4 kv = load_k4(reinterpret_cast<const float *>(base + OFF_KC +
                                                                          (U & 1u) * (OKR * 16)) +
                                              row * DK, DK);
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.v_empty[U & 1u]);
                const F2 kd[4] = {f2_dup(kv.x), f2_dup(kv.y), f2_dup(kv.z), f2_dup(kv.w)};
                F2 dk2[4] = {f2_dup(0.f), f2_dup(0.f), f2_dup(0.f), f2_dup(0.f)};
                // eight of this thread's queries (chunk c4 of its 32, one 16-byte
                // chunk of its P^T row), their G^T values in g; the diagonal tile
                // (queries of the key tile itself) masks i < j
                auto chunk = [&](uint32_t rsa, const uint32_t (&g)[8], uint32_t pb, int c4,
                                 auto masked) {
                    const int qc = OPART * part + 8 * c4;       // first tile column
                    const int c8 = (qc & 63) >> 3;              // chunk in its 64-query K block
                    pb += (uint32_t)(qc >> 6) * P_BLOCK;
                    uint32_t pk[4];
#pragma unroll
                    for (int h4 = 0; h4 < 2; ++h4) {
                        const int q0 = qc + 4 * h4;             // tile column
                        F2 fx[kRecFields][2];                   // field x of queries q0.. in pairs
                        const uint32_t ra = rsa + (uint32_t)q0 * 4u;
#pragma unroll
                        for (int x = 0; x < DK; ++x) f2_lds2(ra + x * OQ * 4, fx[x][0], fx[x][1]);
                        f2_lds2(ra + 4 * OQ * 4, fx[4][0], fx[4][1]);
                        f2_lds2(ra + 5 * OQ * 4, fx[5][0], fx[5][1]);
                        if constexpr (WK == kWSoftmax) f2_lds2(ra + 6 * OQ * 4, fx[6][0], fx[6][1]);
#pragma unroll
                        for (int e = 0; e < 2; ++e) {    // query pairs (q0 + 2e, +1)
                            const int cc = 4 * h4 + 2 * e;        // within g
                            F2 dqk[4];
                            F2 d2 = f2_dup(0.f);
#pragma unroll
                            for (int x = 0; x < DK; ++x) {
                                dqk[x] = f2_sub(fx[x][e], kd[x]);
                                d2 = x == 0 ? f2_mul(dqk[x], dqk[x]) : f2_fma(dqk[x], dqk[x], d2);
                            }
                            F2 wv;
                            if constexpr (WK == kWCauchy) {
                                wv = f2_rcp_approx(f2_fma(d2, ig2, one2));
                            } else {
                                float d2l, d2h, ml = 0.f, mh = 0.f;
                                f2_unpack(d2, d2l, d2h);
                                if constexpr (WK == kWSoftmax) f2_unpack(fx[6][e], ml, mh);
                                wv = f2_pack(weight_fast<WK>(d2l, ml, ig2s), weight_fast<WK>(d2h, mh, ig2s));
                            }
                            if constexpr (decltype(masked)::value) {
                                const int col = q0 + 2 * e;
                                float wl, wh;
                                f2_unpack(wv, wl, wh);
                                wv = f2_pack(col >= row ? wl : 0.f, col + 1 >= row ? wh : 0.f);
                            }
                            const F2 inv_s = fx[4][e], ngbs = fx[5][e];
                            const F2 gv = f2_pack_u(g[cc], g[cc + 1]);
                            const F2 aw = f2_mul(wv, inv_s);
                            const F2 dldw = f2_fma(gv, inv_s, ngbs);
                            F2 ndw;
                            if constexpr (WK == kWSoftmax) ndw = f2_mul(wv, two_ig2);
                            else if constexpr (WK == kWInvEuclid) ndw = f2_mul(f2_mul(wv, wv), wv);
                            else ndw = f2_mul(wv, wv);
                            const F2 coef = f2_mul(dldw, ndw);
#pragma unroll
                            for (int x = 0; x < DK; ++x) dk2[x] = f2_fma(coef, dqk[x], dk2[x]);
                            pk[2 * h4 + e] = f2_bf16x2(aw);
                        }
                    }
                    const uint32_t addr = pb + (uint32_t)((c8 ^ (row & 7)) << 4);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr),
                                 "r"(pk[0]), "r"(pk[1]), "r"(pk[2]), "r"(pk[3])
                                 : "memory");
                };
                // a tile: G^T read 8 columns at a time, the next load in flight
                // while a chunk is computed; the buffer goes back to the MMA once
                // the last load is complete
                auto tile = [&](uint32_t rsa, uint32_t ga, uint32_t pb, uint64_t *gempty,
                                auto masked) {
                    uint32_t gb[2][8];
                    tmem_ld8(ga, gb[0]);
                    tmem_ld_wait_tied(gb[0]);
#pragma unroll
                    for (int c4 = 0; c4 < OCH; ++c4) {
                        if (c4 + 1 < OCH) tmem_ld8(ga + 8u * (c4 + 1), gb[(c4 + 1) & 1]);
                        chunk(rsa, gb[c4 & 1], pb, c4, masked);
                        if (c4 + 1 < OCH) tmem_ld_wait_tied(gb[(c4 + 1) & 1]);
                        if (c4 + 2 == OCH || OCH == 1) {     // every column of the buffer read
                            tc05_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(gempty);
                        }
                    }
                };
                for (int t = 0; t < ntile; ++t) {
                    const uint32_t Tt = T + t, s = Tt % OSTG, b = Tt & 1u;
                    bool okw = own_wait(sh, &sh.g_full[b], (Tt >> 1) & 1u, status) &&
                               own_wait(sh, &sh.p_empty[b], ((Tt >> 1) & 1u) ^ 1u, status) &&
                               own_wait(sh, &sh.d_full[s], (Tt / OSTG) & 1u, status);
                    if (!__all_sync(kFull, okw)) { ok = false; break; }
                    tc05_fence_after();
                    const uint32_t ga = tl + b * OQ + (uint32_t)(OPART * part);
                    const uint32_t rsa = sR + s * (uint32_t)sizeof(OwnRecs);
                    if (t == 0) tile(rsa, ga, sP + b * P_BYTES, &sh.g_empty[b], std::true_type{});
                    else tile(rsa, ga, sP + b * P_BYTES, &sh.g_empty[b], std::false_type{});
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sh.p_full[b]);
                    if (t == 0 && pend) {
                        if (!(ok = epilogue())) break;
                        pend = false;
                    }
                }
                if (!ok) break;
                T += ntile;
                // this unit's dk part for the deferred epilogue, into buffer
                // U & 1 once the unit two back has been read from it
                float dks[4];
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    float lo, hi;
                    f2_unpack(dk2[x], lo, hi);
                    dks[x] = lo + hi;
                }
                {
                    const uint32_t a = U & 1u;
                    bool okw = own_wait(sh, &sh.red_free[a], ((U >> 1) & 1u) ^ 1u, status);
                    if (!__all_sync(kFull, okw)) { ok = false; break; }
                    red[(a * OPARTS + part) * OKR + row] = make_float4(dks[0], dks[1], dks[2], dks[3]);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sh.red_full[a]);
                }
                pend = true;
                pU = U;
                pgj = gj;
            }
        }
        if (ok && pend) ok = epilogue();
    }
    __syncwarp();
    tc05_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc05_fence_after();
        tmem_dealloc(tmem, TM_COLS);
    }
}

template <int DK, int WK>
cudaError_t launch_own(const Prob &p, const CUtensorMap &vmap, const CUtensorMap &dmap,
                       const float *k, const float *gamma, const void *rec, float *own_dv,
                       float *own_dk, int32_t *status, cudaStream_t st) {
    static PerDeviceOnce smem_once;          // run once per device, outside any capture
    cudaError_t e = smem_once.run([] {
        return cudaFuncSetAttribute(bwd_key_own_tc05<DK, WK>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kOwnSmem);
    });
    int dev = 0, sms = 0;
    if (e == cudaSuccess) e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int64_t units = p.S * (int64_t)(p.N / p.C) * (p.C / OKR);
    const int64_t pairs = (units + 1) / 2;
    const unsigned grid = (unsigned)(pairs < sms ? pairs : sms);
    bwd_key_own_tc05<DK, WK><<<grid, OTHREADS, kOwnSmem, st>>>(
        vmap, dmap, k, gamma, static_cast<const QRec *>(rec), own_dv, own_dk, p.N, p.H, p.C, units,
        status);
    return cudaGetLastError();
}

template <int WK>
cudaError_t launch_own_dk(const Prob &p, const CUtensorMap &vmap, const CUtensorMap &dmap,
                          const float *k, const float *gamma, const void *rec, float *own_dv,
                          float *own_dk, int32_t *status, cudaStream_t st) {
    switch (p.dK) {
        case 1: return launch_own<1, WK>(p, vmap, dmap, k, gamma, rec, own_dv, own_dk, status, st);
        case 2: return launch_own<2, WK>(p, vmap, dmap, k, gamma, rec, own_dv, own_dk, status, st);
        case 3: return launch_own<3, WK>(p, vmap, dmap, k, gamma, rec, own_dv, own_dk, status, st);
        default: return launch_own<4, WK>(p, vmap, dmap, k, gamma, rec, own_dv, own_dk, status, st);
    }
}

}  // namespace

bool bwd_own_tc05_supported(const Prob &p) {
    return p.vdt == ZETA_BF16 && p.dV == ODV && p.dK <= 4 && p.C % OKR == 0 && p.N % p.C == 0 &&
           p.S * (int64_t)p.N <= INT32_MAX && p.H <= kMaxHeads;
}

cudaError_t launch_bwd_key_own_tc05(const Prob &p, const float *k, const void *v,
                                    const float *gamma, const void *dout, const void *rec,
                                    float *own_dv, float *own_dk, int32_t *status,
                                    cudaStream_t st) {
    const int64_t rows = p.S * (int64_t)p.N;
    // the copies want 16-byte aligned sources: otherwise (or with no tensor-map
    // encoder) the key kernel computes the own-chunk block itself
    auto misaligned = [](const void *x) { return (reinterpret_cast<uintptr_t>(x) & 15u) != 0; };
    if (!tensor_map_encoder() || misaligned(k) || misaligned(v) || misaligned(dout))
        return cudaErrorNotSupported;
    CUtensorMap vmap, dmap;
    if (!bf16_map(&vmap, v, rows, ODV, 64, OKR) || !bf16_map(&dmap, dout, rows, ODV, 64, OQ))
        return cudaErrorNotSupported;
    if (p.wk == kWSoftmax)
        return launch_own_dk<kWSoftmax>(p, vmap, dmap, k, gamma, rec, own_dv, own_dk, status, st);
    if (p.wk == kWInvEuclid)
        return launch_own_dk<kWInvEuclid>(p, vmap, dmap, k, gamma, rec, own_dv, own_dk, status,
                                          st);
    return launch_own_dk<kWCauchy>(p, vmap, dmap, k, gamma, rec, own_dv, own_dk, status, st);
}

}  // namespace zeta
