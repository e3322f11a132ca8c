// encode.cu -- quantise and bit-interleave every token into a Z-order code.
//
// Passage: OpenReview discussion of "ZETA: Leveraging Z-order Curves for
// Efficient Top-k Attention", reply A2 "Clarification of Binary Expansion and
// Precision": each coordinate is normalised to [0, 1], discretised onto a grid
// of 2^bits cells and the cell indices' bits are interleaved into one integer.
// Coordinate 0 is the most significant bit of every level (the K^1, K^2, K^3
// order of the reply on dimension-ordering asymmetry).
//
// One thread per token.  The work is a few integer operations per 4*d_K bytes
// read, so the kernel runs at copy speed; bit spreading for d_K = 2 and 3 uses
// the usual shift-and-mask ("magic number") dilation, other widths a bit loop.
#include "zorder.cuh"

namespace zeta {
namespace {

template <typename CodeT>
__global__ void encode_kernel(const float *__restrict__ x, CodeT *__restrict__ codes,
                              int64_t ntok, int dK, int bits) {
    const float scale = __int_as_float((126 + bits) << 23);   // 2^(bits-1)
    const float umax = static_cast<float>((1u << bits) - 1u);
    for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < ntok;
         t += (int64_t)gridDim.x * blockDim.x) {
        const float *xt = x + t * dK;
        uint64_t code = 0;
        if (dK == 3) {
            uint32_t u0 = quantise(xt[0], scale, umax);
            uint32_t u1 = quantise(xt[1], scale, umax);
            uint32_t u2 = quantise(xt[2], scale, umax);
            code = (dilate3(u0) << 2) | (dilate3(u1) << 1) | dilate3(u2);
        } else if (dK == 2) {
            uint32_t u0 = quantise(xt[0], scale, umax);
            uint32_t u1 = quantise(xt[1], scale, umax);
            code = (dilate2(u0) << 1) | dilate2(u1);
        } else if (dK == 1) {
            code = quantise(xt[0], scale, umax);
        } else {
            for (int d = 0; d < dK; ++d) {
                uint32_t u = quantise(xt[d], scale, umax);
                const int sh = dK - 1 - d;
                for (int j = 0; j < bits; ++j)
                    code |= static_cast<uint64_t>((u >> j) & 1u) << (j * dK + sh);
            }
        }
        codes[t] = static_cast<CodeT>(code);
    }
}

constexpr int kMaxCurves = 8;

struct CurveAxes {
    int8_t a[kMaxCurves][kMaxDK];
};

// Several curves per token: the cells are computed once, then combined in
// each curve's coordinate order (for d_K = 3, three shifts per curve).
template <typename CodeT>
__global__ void encode_curves_kernel(const float *__restrict__ x, CodeT *__restrict__ codes,
                                     int64_t ntok, int dK, int bits, int curves, CurveAxes ax) {
    const float scale = __int_as_float((126 + bits) << 23);   // 2^(bits-1)
    const float umax = static_cast<float>((1u << bits) - 1u);
    for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < ntok;
         t += (int64_t)gridDim.x * blockDim.x) {
        const float *xt = x + t * dK;
        uint32_t u[kMaxDK];
#pragma unroll
        for (int d = 0; d < kMaxDK; ++d) u[d] = d < dK ? quantise(xt[d], scale, umax) : 0u;
        if (dK == 3) {
            const uint64_t s0 = dilate3(u[0]), s1 = dilate3(u[1]), s2 = dilate3(u[2]);
            for (int m = 0; m < curves; ++m) {
                const int a0 = ax.a[m][0], a1 = ax.a[m][1], a2 = ax.a[m][2];
                const uint64_t c0 = a0 == 0 ? s0 : (a0 == 1 ? s1 : s2);
                const uint64_t c1 = a1 == 0 ? s0 : (a1 == 1 ? s1 : s2);
                const uint64_t c2 = a2 == 0 ? s0 : (a2 == 1 ? s1 : s2);
                codes[m * ntok + t] = static_cast<CodeT>((c0 << 2) | (c1 << 1) | c2);
            }
        } else {
            for (int m = 0; m < curves; ++m) {
                uint64_t code = 0;
                for (int d = 0; d < dK; ++d) {
                    uint32_t v = 0;
#pragma unroll
                    for (int e = 0; e < kMaxDK; ++e) v = e == ax.a[m][d] ? u[e] : v;
                    const int sh = dK - 1 - d;
                    for (int j = 0; j < bits; ++j)
                        code |= static_cast<uint64_t>((v >> j) & 1u) << (j * dK + sh);
                }
                codes[m * ntok + t] = static_cast<CodeT>(code);
            }
        }
    }
}

}  // namespace

cudaError_t launch_encode(const Prob &p, const float *x, void *codes, cudaStream_t st) {
    const int64_t ntok = p.S * p.N;
    const int threads = 256;
    int64_t blocks = (ntok + threads - 1) / threads;
    if (blocks > 152 * 64) blocks = 152 * 64;
    if (p.code64)
        encode_kernel<uint64_t><<<(unsigned)blocks, threads, 0, st>>>(
            x, static_cast<uint64_t *>(codes), ntok, p.dK, p.bits);
    else
        encode_kernel<uint32_t><<<(unsigned)blocks, threads, 0, st>>>(
            x, static_cast<uint32_t *>(codes), ntok, p.dK, p.bits);
    return cudaGetLastError();
}

cudaError_t launch_encode_curves(const Prob &p, const float *x, int curves, const int32_t *axes,
                                 void *codes, cudaStream_t st) {
    CurveAxes ax{};
    for (int m = 0; m < curves; ++m)
        for (int d = 0; d < p.dK; ++d) ax.a[m][d] = static_cast<int8_t>(axes[m * p.dK + d]);
    const int64_t ntok = p.S * p.N;
    const int threads = 256;
    int64_t blocks = (ntok + threads - 1) / threads;
    if (blocks > 152 * 64) blocks = 152 * 64;
    if (p.code64)
        encode_curves_kernel<uint64_t><<<(unsigned)blocks, threads, 0, st>>>(
            x, static_cast<uint64_t *>(codes), ntok, p.dK, p.bits, curves, ax);
    else
        encode_curves_kernel<uint32_t><<<(unsigned)blocks, threads, 0, st>>>(
            x, static_cast<uint32_t *>(codes), ntok, p.dK, p.bits, curves, ax);
    return cudaGetLastError();
}

}  // namespace zeta
