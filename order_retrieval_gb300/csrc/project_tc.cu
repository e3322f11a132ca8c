// project_tc.cu -- the two-layer projection front end fused with the Z-order
// encode, on the Blackwell tensor cores (tcgen05 + TMEM, TMA-fed).
//
// Passage: OpenReview discussion of "ZETA: Leveraging Z-order Curves for
// Efficient Top-k Attention", reply A "LLMs impact the selection of d_K" (a
// two-layer neural network projects the input into the low-dimensional keys),
// and reply A2 "Clarification of Binary Expansion and Precision" (the codes).
// Per head hd and token t (queries and keys each with their own weights):
//   h_f = max(0, W1[hd F + f] . x_t + b1[hd F + f]),   f < F
//   y_c = tanh(W2[hd][c] . h + b2[hd][c]),             c < d_K
// then y is written out and quantised into the token's Morton code.
//
// One CTA computes 128 tokens x 256 hidden units (four heads of F = 64) of one
// projection: the first layer is a K = D contraction on tcgen05.mma (M = 128,
// N = 256, K = 16 per instruction, bf16 in, f32 accumulator in 256 TMEM
// columns).  x and W1 tiles of 64 K-elements (128 bytes, the 128-byte swizzle
// row) are brought by 2-D TMA loads into a three-stage ring; one thread waits
// for a stage, issues its four MMAs and commits them to the stage's "empty"
// barrier, then refills the stage of the previous step.  The epilogue runs on
// all four warps: each thread owns one token (one TMEM lane), reads its 64
// accumulators of a head with tcgen05.ld, applies bias and ReLU, the 64 -> d_K
// second layer from shared memory, tanh, and the quantiser + bit interleave.
// Every wait is bounded; a wait that gives up records ZETA_ERR_DEVICE_TIMEOUT,
// drains the loads in flight (again bounded) and frees the TMEM before exiting.
#include <cudaTypedefs.h>

#include "tc05.cuh"
#include "zorder.cuh"

namespace zeta {
namespace {

constexpr int BM = 128;                   // tokens per CTA
constexpr int BN = 256;                   // hidden units per CTA
constexpr int BK = 64;                    // K elements per stage (128 bytes of bf16)
constexpr int FH = 64;                    // hidden units per head
constexpr int HPC = BN / FH;              // heads per CTA
constexpr int STAGES = 3;
constexpr int PTHREADS = 128;
constexpr uint32_t A_BYTES = BM * BK * 2;
constexpr uint32_t B_BYTES = BN * BK * 2;
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;

struct ProjHead {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t done;
    uint32_t tmem_base;
    int32_t err;
    float b1[BN];
    float w2[HPC][4][FH];
    float b2[HPC][4];
};

constexpr size_t kProjSmem = 1024 + STAGES * STAGE_BYTES + sizeof(ProjHead);

template <typename CodeT>
__global__ void __launch_bounds__(PTHREADS, 1)
project_encode_tc(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
                  const float *__restrict__ b1, const float *__restrict__ w2,
                  const float *__restrict__ b2, float *__restrict__ qo, float *__restrict__ ko,
                  CodeT *__restrict__ qc, CodeT *__restrict__ kc, int64_t M, int N, int H, int dK,
                  int D, int bits, int32_t *status) {
    extern __shared__ unsigned char dsm[];
    unsigned char *base = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(dsm) + 1023) & ~uintptr_t(1023));
    ProjHead &sh = *reinterpret_cast<ProjHead *>(base + STAGES * STAGE_BYTES);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t m0 = (int64_t)blockIdx.x * BM;
    const int ct = blockIdx.y;
    const int tiles_per_proj = H * FH / BN;
    const int pr = ct / tiles_per_proj;               // 0: queries, 1: keys
    const int h0 = (ct % tiles_per_proj) * HPC;
    const int KB = D / BK;

    for (int t = tid; t < BN; t += PTHREADS) sh.b1[t] = b1[((int64_t)pr * H + h0) * FH + t];
    for (int t = tid; t < HPC * 4 * FH; t += PTHREADS) {
        const int hh = t / (4 * FH), c = (t / FH) & 3, f = t % FH;
        sh.w2[hh][c][f] = c < dK ? w2[(((int64_t)pr * H + h0 + hh) * dK + c) * FH + f] : 0.f;
    }
    if (tid < HPC * 4) {
        const int hh = tid >> 2, c = tid & 3;
        sh.b2[hh][c] = c < dK ? b2[((int64_t)pr * H + h0 + hh) * dK + c] : 0.f;
    }
    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&sh.full[s], 1);
            mbar_init(&sh.empty[s], 1);
        }
        mbar_init(&sh.done, 1);
        sh.err = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&sh.tmem_base, BN);
        tmem_relinquish();
    }
    tc05_fence_before();
    __syncthreads();
    tc05_fence_after();
    const uint32_t tmem = sh.tmem_base;

    // ------------------------------------------------ producer + MMA issue ---
    if (tid == 0) {
        auto load = [&](int kb) {
            const int s = kb % STAGES;
            unsigned char *sa = base + s * STAGE_BYTES;
            mbar_arrive_expect_tx(&sh.full[s], STAGE_BYTES);
            tma_load_2d(sa, &xmap, kb * BK, (int)m0, &sh.full[s]);
            tma_load_2d(sa + A_BYTES, &wmap, kb * BK, ct * BN, &sh.full[s]);
        };
        const int pre = KB < STAGES ? KB : STAGES;
        for (int kb = 0; kb < pre; ++kb) load(kb);
        int issued = pre, consumed = 0;
        bool ok = true;
        constexpr uint32_t idesc = idesc_bf16_f32(BM, BN);
        for (int kb = 0; kb < KB; ++kb) {
            const int s = kb % STAGES;
            if (!mbar_wait_bounded(&sh.full[s], (uint32_t)(kb / STAGES) & 1u)) {
                ok = false;
                break;
            }
            consumed = kb + 1;
            tc05_fence_after();
            const uint32_t sa = smem_u32(base + s * STAGE_BYTES);
            const uint64_t ad = sdesc_k128(sa), bd = sdesc_k128(sa + A_BYTES);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)   // 32 bytes of K per instruction
                umma_bf16(tmem, ad + 2u * kk, bd + 2u * kk, idesc, (kb | kk) != 0);
            umma_commit(&sh.empty[s]);
            const int kp = kb - 1;                  // refill the previous step's stage
            if (kp >= 0 && kp + STAGES < KB) {
                if (!mbar_wait_bounded(&sh.empty[kp % STAGES], (uint32_t)(kp / STAGES) & 1u)) {
                    ok = false;
                    break;
                }
                load(kp + STAGES);
                issued = kp + STAGES + 1;
            }
        }
        if (ok) {
            umma_commit(&sh.done);
        } else {
            sh.err = 1;
            set_status(status, ZETA_ERR_DEVICE_TIMEOUT);
            for (int kb = consumed; kb < issued; ++kb)      // loads still in flight
                mbar_wait_bounded(&sh.full[kb % STAGES], (uint32_t)(kb / STAGES) & 1u);
        }
    }
    __syncwarp();
    __syncthreads();

    // --------------------------------------------------------- epilogue ---
    bool good = sh.err == 0;
    if (good && !mbar_wait_bounded(&sh.done, 0)) {
        good = false;
        set_status(status, ZETA_ERR_DEVICE_TIMEOUT);
    }
    tc05_fence_after();
    good = __all_sync(kFull, good);
    if (good) {
        const int row = warp * 32 + lane;                  // this thread's TMEM lane
        const int64_t m = m0 + row;
        const bool valid = m < M;
        const int64_t bsl = valid ? m / N : 0;
        const int n = valid ? (int)(m % N) : 0;
        float *outp = pr == 0 ? qo : ko;
        CodeT *codep = pr == 0 ? qc : kc;
        const float scale = __int_as_float((126 + bits) << 23);   // 2^(bits-1)
        const float umax = static_cast<float>((1u << bits) - 1u);
        for (int hh = 0; hh < HPC; ++hh) {
            float y[4] = {sh.b2[hh][0], sh.b2[hh][1], sh.b2[hh][2], sh.b2[hh][3]};
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t r[32];
                tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(hh * FH + half * 32), r);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int f = half * 32 + j;
                    const float hv = fmaxf(__uint_as_float(r[j]) + sh.b1[hh * FH + f], 0.f);
#pragma unroll
                    for (int c = 0; c < 4; ++c) y[c] = __fmaf_rn(sh.w2[hh][c][f], hv, y[c]);
                }
            }
            if (valid) {
                const int64_t tok = (bsl * H + h0 + hh) * (int64_t)N + n;
                uint32_t u[4];
                for (int c = 0; c < dK; ++c) {
                    const float yc = tanhf(y[c]);
                    outp[tok * dK + c] = yc;
                    u[c] = quantise(yc, scale, umax);
                }
                uint64_t code = 0;
                if (dK == 3) {
                    code = morton3(u[0], u[1], u[2]);
                } else {
                    for (int c = 0; c < dK; ++c)
                        for (int j = 0; j < bits; ++j)
                            code |= static_cast<uint64_t>((u[c] >> j) & 1u) << (j * dK + dK - 1 - c);
                }
                codep[tok] = static_cast<CodeT>(code);
            }
        }
    }
    tc05_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc05_fence_after();
        tmem_dealloc(tmem, BN);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &qr) != cudaSuccess ||
            qr != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// Row-major bf16 matrix [rows, cols] as a 2-D TMA map with a (64 x box_rows)
// box and the 128-byte swizzle.
bool bf16_map(CUtensorMap *map, const void *ptr, int64_t rows, int64_t cols, int box_rows) {
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1u, 1u};
    return tensor_map_encoder()(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr),
                                dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool project_tc_supported(const Prob &p, int D, int F) {
    return F == FH && D >= BK && D % BK == 0 && (p.H * FH) % BN == 0 && p.dK <= 4 &&
           p.S * (int64_t)p.N <= INT32_MAX && tensor_map_encoder() != nullptr;
}

cudaError_t launch_project_tc(const Prob &p, int D, const void *x, const void *w1,
                              const float *b1, const float *w2, const float *b2, float *q,
                              float *k, void *q_codes, void *k_codes, int32_t *status,
                              cudaStream_t st) {
    const int64_t M = (int64_t)p.B * p.N;
    CUtensorMap xmap, wmap;
    if (!bf16_map(&xmap, x, M, D, BM) || !bf16_map(&wmap, w1, 2LL * p.H * FH, D, BN))
        return cudaErrorInvalidValue;
    const dim3 grid((unsigned)((M + BM - 1) / BM), (unsigned)(2 * p.H * FH / BN));
    if (p.code64) {
        static bool attr64 = false;
        if (!attr64) {
            cudaError_t e = cudaFuncSetAttribute(project_encode_tc<uint64_t>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)kProjSmem);
            if (e != cudaSuccess) return e;
            attr64 = true;
        }
        project_encode_tc<uint64_t><<<grid, PTHREADS, kProjSmem, st>>>(
            xmap, wmap, b1, w2, b2, q, k, static_cast<uint64_t *>(q_codes),
            static_cast<uint64_t *>(k_codes), M, p.N, p.H, p.dK, D, p.bits, status);
    } else {
        static bool attr32 = false;
        if (!attr32) {
            cudaError_t e = cudaFuncSetAttribute(project_encode_tc<uint32_t>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)kProjSmem);
            if (e != cudaSuccess) return e;
            attr32 = true;
        }
        project_encode_tc<uint32_t><<<grid, PTHREADS, kProjSmem, st>>>(
            xmap, wmap, b1, w2, b2, q, k, static_cast<uint32_t *>(q_codes),
            static_cast<uint32_t *>(k_codes), M, p.N, p.H, p.dK, D, p.bits, status);
    }
    return cudaGetLastError();
}

}  // namespace zeta
