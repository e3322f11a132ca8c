// project_tc.cu -- the two-layer projection front end fused with the Z-order
// encode, on the Blackwell tensor cores (tcgen05 + TMEM, TMA-fed).
//
// Passage: OpenReview discussion of "ZETA: Leveraging Z-order Curves for
// Efficient Top-k Attention", reply A "LLMs impact the selection of d_K" (the
// low-dimensional keys come out of a small network of two layers),
// and reply A2 "Clarification of Binary Expansion and Precision" (the codes).
// Per head hd and token t (queries and keys each with their own weights):
//   h_f = max(0, W1[hd F + f] . x_t + b1[hd F + f]),   f < F
//   y_c = tanh(W2[hd][c] . h + b2[hd][c]),             c < d_K
// then y is written out and quantised into the token's Morton code.
//
// Work unit: 128 tokens x 256 hidden units (four heads of F = 64) of one
// projection; the first layer is a K = D contraction on tcgen05.mma (M = 128,
// N = 256, K = 16 per instruction, bf16 in, f32 accumulator in TMEM).  The
// kernel is persistent (one CTA per SM walking the units, the four units of a
// token tile next to each other so the x tile is reused from L2) and
// warp-specialised:
//   warp 0    TMA producer: x and W1 tiles of 64 K-elements (128 bytes, the
//             128-byte swizzle row) into a four-stage ring;
//   warp 1    MMA issuer (one thread) and owner of the TMEM allocation: two
//             256-column accumulators, so a unit's MMAs run while the previous
//             unit's epilogue drains the other accumulator;
//   warps 2-9 epilogue: two warps per TMEM lane quarter, each taking two of
//             the unit's four heads; a thread owns one token (one TMEM lane),
//             reads its 64 accumulators of a head with tcgen05.ld, applies bias
//             and ReLU, the 64 -> d_K second layer (weights staged in shared
//             memory, packed f32x2 FMAs), tanh, and the quantiser + bit
//             interleave.
// Hand-offs are mbarriers: full/empty per ring stage (TMA -> MMA -> TMA), and
// full/empty per accumulator (MMA commit -> epilogue -> MMA).  Every wait is
// bounded; a wait that gives up records ZETA_ERR_DEVICE_TIMEOUT and raises an
// abort flag that ends every role's loop; the producer then waits (bounded)
// for its loads in flight and the MMA thread for its MMAs before the TMEM is
// freed.
#include "tc05.cuh"
#include "tmap.cuh"
#include "zorder.cuh"

namespace zeta {
namespace {

constexpr int BM = 128;                   // tokens per unit
constexpr int BN = 256;                   // hidden units per unit
constexpr int BK = 64;                    // K elements per stage (128 bytes of bf16)
constexpr int FH = 64;                    // hidden units per head
constexpr int HPC = BN / FH;              // heads per unit
constexpr int STAGES = 4;
constexpr int EPI_WARPS = 8;
constexpr int PTHREADS = 64 + 32 * EPI_WARPS;   // producer, MMA, epilogue warps
constexpr int MAX_H = 8;
constexpr uint32_t A_BYTES = BM * BK * 2;
constexpr uint32_t B_BYTES = BN * BK * 2;
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t TMEM_COLS = 2 * BN;    // two accumulators

struct ProjHead {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int32_t abort;
};

// Second-layer parameters of both projections, staged once per CTA.
struct ProjParams {
    float b1[2][MAX_H * FH];
    float4 w2[2][MAX_H][FH];              // (W2[0][f], .. W2[3][f]), d_K padded with zeros
    float4 b2[2][MAX_H];
};

constexpr size_t kProjSmem = 1024 + STAGES * STAGE_BYTES + sizeof(ProjHead) + sizeof(ProjParams);

__device__ __forceinline__ bool aborted(const ProjHead &sh) {
    return *reinterpret_cast<const volatile int32_t *>(&sh.abort) != 0;
}

__device__ __forceinline__ bool wait_or_abort(ProjHead &sh, uint64_t *bar, uint32_t parity,
                                              int32_t *status) {
    if (mbar_wait_bounded(bar, parity)) return true;
    *reinterpret_cast<volatile int32_t *>(&sh.abort) = 1;
    set_status(status, ZETA_ERR_DEVICE_TIMEOUT);
    return false;
}

template <typename CodeT, int DK>
__global__ void __launch_bounds__(PTHREADS, 1)
project_encode_tc(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
                  const float *__restrict__ b1, const float *__restrict__ w2,
                  const float *__restrict__ b2, float *__restrict__ qo, float *__restrict__ ko,
                  CodeT *__restrict__ qc, CodeT *__restrict__ kc, int64_t M, int N, int H, int D,
                  int bits, int32_t *status) {
    extern __shared__ unsigned char dsm[];
    unsigned char *base = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(dsm) + 1023) & ~uintptr_t(1023));
    ProjHead &sh = *reinterpret_cast<ProjHead *>(base + STAGES * STAGE_BYTES);
    ProjParams &pp = *reinterpret_cast<ProjParams *>(base + STAGES * STAGE_BYTES +
                                                    sizeof(ProjHead));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n_ct = 2 * H * FH / BN;                 // units per token tile
    const int64_t n_mt = (M + BM - 1) / BM;
    const int64_t units = n_mt * n_ct;
    const int KB = D / BK;

    for (int t = tid; t < 2 * H * FH; t += PTHREADS) pp.b1[t / (H * FH)][t % (H * FH)] = b1[t];
    for (int t = tid; t < 2 * H * 4 * FH; t += PTHREADS) {
        const int pr = t / (H * 4 * FH), hd = (t / (4 * FH)) % H, c = (t / FH) & 3, f = t % FH;
        reinterpret_cast<float *>(&pp.w2[pr][hd][f])[c] =
            c < DK ? w2[(((int64_t)pr * H + hd) * DK + c) * FH + f] : 0.f;
    }
    for (int t = tid; t < 2 * H * 4; t += PTHREADS) {
        const int pr = t / (H * 4), hd = (t / 4) % H, c = t & 3;
        reinterpret_cast<float *>(&pp.b2[pr][hd])[c] =
            c < DK ? b2[((int64_t)pr * H + hd) * DK + c] : 0.f;
    }
    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&sh.full[s], 1);
            mbar_init(&sh.empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&sh.acc_full[a], 1);
            mbar_init(&sh.acc_empty[a], EPI_WARPS);   // one arrive per epilogue warp
        }
        mbar_init(&sh.drain, 1);
        sh.abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&sh.tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    tc05_fence_before();
    __syncthreads();
    tc05_fence_after();
    const uint32_t tmem = sh.tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------ producer ---
        if (lane == 0) {
            uint32_t it = 0;
            for (int64_t u = blockIdx.x; u < units && !aborted(sh); u += gridDim.x) {
                const int mt = (int)(u / n_ct), ct = (int)(u % n_ct);
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const uint32_t s = it % STAGES;
                    if (!wait_or_abort(sh, &sh.empty[s], ((it / STAGES) & 1u) ^ 1u, status)) break;
                    unsigned char *sa = base + s * STAGE_BYTES;
                    mbar_arrive_expect_tx(&sh.full[s], STAGE_BYTES);
                    tma_load_2d(sa, &xmap, kb * BK, mt * BM, &sh.full[s]);
                    tma_load_2d(sa + A_BYTES, &wmap, kb * BK, ct * BN, &sh.full[s]);
                }
            }
            if (aborted(sh)) {
                // the last load into each stage completes after all earlier ones
                for (uint32_t s = 0; s < STAGES; ++s) {
                    if (it <= s) continue;
                    const uint32_t last = it - 1 - ((it - 1 + STAGES - s) % STAGES);
                    mbar_wait_bounded(&sh.full[s], (last / STAGES) & 1u);
                }
            }
        }
    } else if (warp == 1) {
        // --------------------------------------------------------- MMA ---
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(BM, BN);
            uint32_t it = 0, lt = 0;
            bool issued = false;
            for (int64_t u = blockIdx.x; u < units && !aborted(sh); u += gridDim.x, ++lt) {
                const uint32_t a = lt & 1u;
                if (!wait_or_abort(sh, &sh.acc_empty[a], ((lt >> 1) & 1u) ^ 1u, status)) break;
                tc05_fence_after();
                const uint32_t dt = tmem + a * BN;
                bool ok = true;
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const uint32_t s = it % STAGES;
                    if (!wait_or_abort(sh, &sh.full[s], (it / STAGES) & 1u, status)) {
                        ok = false;
                        break;
                    }
                    tc05_fence_after();
                    const uint32_t sa = smem_u32(base + s * STAGE_BYTES);
                    const uint64_t ad = sdesc_k128(sa), bd = sdesc_k128(sa + A_BYTES);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)   // 32 bytes of K per instruction
                        umma_bf16(dt, ad + 2u * kk, bd + 2u * kk, idesc, (kb | kk) != 0);
                    issued = true;
                    umma_commit(&sh.empty[s]);
                }
                if (!ok) break;
                umma_commit(&sh.acc_full[a]);
            }
            if (issued && aborted(sh)) {
                umma_commit(&sh.drain);
                mbar_wait_bounded(&sh.drain, 0);
            }
        }
    } else {
        // ---------------------------------------------------- epilogue ---
        const int quarter = warp & 3;                     // TMEM lanes 32*quarter ..
        const int hhalf = (warp - 2) >> 2;                // heads 2*hhalf, 2*hhalf + 1
        const int row = quarter * 32 + lane;
        const float scale = __int_as_float((126 + bits) << 23);   // 2^(bits-1)
        const float umax = static_cast<float>((1u << bits) - 1u);
        uint32_t lt = 0;
        for (int64_t u = blockIdx.x; u < units; u += gridDim.x, ++lt) {
            if (__any_sync(kFull, aborted(sh))) break;
            const uint32_t a = lt & 1u;
            const bool ok = wait_or_abort(sh, &sh.acc_full[a], (lt >> 1) & 1u, status);
            if (!__all_sync(kFull, ok)) break;
            tc05_fence_after();
            const int mt = (int)(u / n_ct), ct = (int)(u % n_ct);
            const int pr = ct / (n_ct / 2);               // 0: queries, 1: keys
            const int h0 = (ct % (n_ct / 2)) * HPC;
            const int64_t m = (int64_t)mt * BM + row;
            const bool valid = m < M;
            const int64_t bsl = valid ? m / N : 0;
            const int n = valid ? (int)(m % N) : 0;
            float *outp = pr == 0 ? qo : ko;
            CodeT *codep = pr == 0 ? qc : kc;
            for (int hq = 0; hq < HPC / 2; ++hq) {
                const int hh = hhalf * (HPC / 2) + hq;
                const int hd = h0 + hh;
                uint32_t r0[32], r1[32];
                const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + a * BN +
                                       (uint32_t)(hh * FH);
                tmem_ld32(taddr, r0);
                tmem_ld32(taddr + 32, r1);
                tmem_ld_wait();
                const float4 bz = pp.b2[pr][hd];
                float2 y01 = make_float2(bz.x, bz.y), y23 = make_float2(bz.z, bz.w);
                const float4 *bb = reinterpret_cast<const float4 *>(pp.b1[pr] + hd * FH);
                const float4 *ww = pp.w2[pr][hd];
#pragma unroll
                for (int f4 = 0; f4 < FH / 4; ++f4) {
                    const float4 b4 = bb[f4];
                    const float bv[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int f = f4 * 4 + e;
                        const float acc = __uint_as_float(f < 32 ? r0[f] : r1[f - 32]);
                        const float2 hv = dup2(fmaxf(acc + bv[e], 0.f));
                        const float4 w = ww[f];
                        y01 = fma2(make_float2(w.x, w.y), hv, y01);
                        if constexpr (DK > 2) y23 = fma2(make_float2(w.z, w.w), hv, y23);
                    }
                }
                const float y[4] = {y01.x, y01.y, y23.x, y23.y};
                if (valid) {
                    const int64_t tok = (bsl * H + hd) * (int64_t)N + n;
                    uint32_t ucell[4];
#pragma unroll
                    for (int c = 0; c < DK; ++c) {
                        const float yc = tanhf(y[c]);
                        outp[tok * DK + c] = yc;
                        ucell[c] = quantise(yc, scale, umax);
                    }
                    uint64_t code = 0;
                    if constexpr (DK == 3) {
                        code = morton3(ucell[0], ucell[1], ucell[2]);
                    } else {
#pragma unroll
                        for (int c = 0; c < DK; ++c)
                            for (int j = 0; j < bits; ++j)
                                code |= static_cast<uint64_t>((ucell[c] >> j) & 1u)
                                        << (j * DK + DK - 1 - c);
                    }
                    codep[tok] = static_cast<CodeT>(code);
                }
            }
            tc05_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.acc_empty[a]);
        }
    }
    __syncwarp();
    tc05_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc05_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

template <typename CodeT, int DK>
cudaError_t launch_proj(const Prob &p, int D, const CUtensorMap &xmap, const CUtensorMap &wmap,
                        const float *b1, const float *w2, const float *b2, float *q, float *k,
                        void *q_codes, void *k_codes, int32_t *status, cudaStream_t st) {
    static PerDeviceOnce smem_once;
    cudaError_t e = smem_once.run([] {
        return cudaFuncSetAttribute(project_encode_tc<CodeT, DK>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kProjSmem);
    });
    int dev = 0, sms = 0;
    if (e == cudaSuccess) e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int64_t M = (int64_t)p.B * p.N;
    const int64_t units = (M + BM - 1) / BM * (2 * p.H * FH / BN);
    const unsigned grid = (unsigned)(units < sms ? units : sms);
    project_encode_tc<CodeT, DK><<<grid, PTHREADS, kProjSmem, st>>>(
        xmap, wmap, b1, w2, b2, q, k, static_cast<CodeT *>(q_codes), static_cast<CodeT *>(k_codes),
        M, p.N, p.H, D, p.bits, status);
    return cudaGetLastError();
}

template <typename CodeT>
cudaError_t launch_proj_dk(const Prob &p, int D, const CUtensorMap &xmap,
                           const CUtensorMap &wmap, const float *b1, const float *w2,
                           const float *b2, float *q, float *k, void *qc, void *kc,
                           int32_t *status, cudaStream_t st) {
    switch (p.dK) {
        case 1: return launch_proj<CodeT, 1>(p, D, xmap, wmap, b1, w2, b2, q, k, qc, kc, status, st);
        case 2: return launch_proj<CodeT, 2>(p, D, xmap, wmap, b1, w2, b2, q, k, qc, kc, status, st);
        case 3: return launch_proj<CodeT, 3>(p, D, xmap, wmap, b1, w2, b2, q, k, qc, kc, status, st);
        default: return launch_proj<CodeT, 4>(p, D, xmap, wmap, b1, w2, b2, q, k, qc, kc, status, st);
    }
}

}  // namespace

bool project_tc_supported(const Prob &p, int D, int F) {
    return F == FH && D >= BK && D % BK == 0 && (p.H * FH) % BN == 0 && p.H <= MAX_H &&
           p.dK <= 4 && p.S * (int64_t)p.N <= INT32_MAX && tensor_map_encoder() != nullptr;
}

cudaError_t launch_project_tc(const Prob &p, int D, const void *x, const void *w1,
                              const float *b1, const float *w2, const float *b2, float *q,
                              float *k, void *q_codes, void *k_codes, int32_t *status,
                              cudaStream_t st) {
    const int64_t M = (int64_t)p.B * p.N;
    CUtensorMap xmap, wmap;
    if (!bf16_map(&xmap, x, M, D, BK, BM) || !bf16_map(&wmap, w1, 2LL * p.H * FH, D, BK, BN))
        return cudaErrorInvalidValue;
    if (p.code64)
        return launch_proj_dk<uint64_t>(p, D, xmap, wmap, b1, w2, b2, q, k, q_codes, k_codes,
                                        status, st);
    return launch_proj_dk<uint32_t>(p, D, xmap, wmap, b1, w2, b2, q, k, q_codes, k_codes, status,
                                    st);
}

}  // namespace zeta
