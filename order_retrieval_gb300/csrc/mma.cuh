// mma.cuh -- inline-PTX helpers shared by the tensor-core kernels:
// cp.async staging, ldmatrix, mma.sync m16n8k16 (bf16 in, f32 accumulate),
// streaming 32-byte loads and bf16 packing.
#pragma once

#include "common.cuh"

namespace zeta {

// Shared-memory tiles of 64 rows x 64 bf16 (128-byte rows) are stored with the
// 16-byte chunk c of row r at chunk position c ^ (r & 7), so the eight row
// addresses of every ldmatrix hit eight different bank groups.
__device__ __forceinline__ int swz(int row, int chunk) { return row * 64 + ((chunk ^ (row & 7)) * 8); }

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
                 "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, "
        "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Transpose of an 8x8 b16 matrix held one 32-bit pair per lane (lane L: row
// L / 4, columns 2 (L % 4), +1) into the same layout.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(d) : "r"(a));
    return d;
}

// 32-byte load through the non-coherent path without L1 allocation (gathered
// rows are used once by the loading warp): two adjacent 16-byte slices at a
// 32-byte aligned address in one 256-bit access; zeros where `ok` is false.
__device__ __forceinline__ void ld_stream32(const void *p, bool ok, uint4 &a, uint4 &b) {
    a = make_uint4(0u, 0u, 0u, 0u);
    b = a;
    asm volatile(
        "{\n .reg .pred q;\n setp.ne.b32 q, %9, 0;\n"
        " @q ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n}\n"
        : "+r"(a.x), "+r"(a.y), "+r"(a.z), "+r"(a.w), "+r"(b.x), "+r"(b.y), "+r"(b.z), "+r"(b.w)
        : "l"(p), "r"((int)ok));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ float4 load_k4(const float *row, int dK) {
    return make_float4(row[0], dK > 1 ? row[1] : 0.f, dK > 2 ? row[2] : 0.f,
                       dK > 3 ? row[3] : 0.f);
}

}  // namespace zeta

namespace zeta {

// ------------------------------------------------------------- mbarrier ---

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count));
}

// Make barrier initialisation visible to the asynchronous (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait for the barrier phase with an iteration limit; false when it gave up.
constexpr uint32_t kWaitLimit = 1u << 22;
__device__ __forceinline__ bool mbar_wait_limit(uint64_t *bar, uint32_t parity, uint32_t limit) {
    for (uint32_t it = 0; it < limit; ++it)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity) {
    return mbar_wait_limit(bar, parity, kWaitLimit);
}

// Cauchy weight with CUDA's fast division intrinsic (documented error of at
// most 2 ulp here, as 1 <= 1 + d2/gamma^2); used where the weight feeds a sum.
__device__ __forceinline__ float cauchy_w_fast(float d2, float inv_g2) {
    return __fdividef(1.0f, __fmaf_rn(d2, inv_g2, 1.0f));
}

}  // namespace zeta

namespace zeta {

// ------------------------------------------- packed float32x2 arithmetic ---
// Two independent float32 lanes per instruction (Blackwell f32x2 forms),
// each rounded exactly as the scalar operation would be.

__device__ __forceinline__ uint64_t f2u(float2 a) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a.x), "f"(a.y));
    return r;
}
__device__ __forceinline__ float2 u2f(uint64_t r) {
    float2 a;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a.x), "=f"(a.y) : "l"(r));
    return a;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2u(a)), "l"(f2u(b)));
    return u2f(r);
}
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2u(a)), "l"(f2u(b)));
    return u2f(r);
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2u(a)), "l"(f2u(b)));
    return u2f(r);
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(f2u(a)), "l"(f2u(b)), "l"(f2u(c)));
    return u2f(r);
}
__device__ __forceinline__ float2 dup2(float x) { return make_float2(x, x); }

// Cauchy weights of two (query, key) pairs at once: d2 holds both squared
// distances; the reciprocals stay scalar (fast division intrinsic).
__device__ __forceinline__ float2 cauchy_w2(float2 d2, float2 inv_g2) {
    const float2 t = fma2(d2, inv_g2, dup2(1.0f));
    return make_float2(__fdividef(1.0f, t.x), __fdividef(1.0f, t.y));
}

// Weight kernels (common.cuh) with fast intrinsics, for weights that feed sums:
// the Cauchy reciprocal by __fdividef, the softmax exponential by __expf
// (m = the query's current shift), inverse Euclidean by rsqrtf.
template <int WK>
__device__ __forceinline__ float weight_fast(float d2, float m, float inv_g2) {
    if constexpr (WK == kWSoftmax) return __expf((m - d2) * inv_g2);
    else if constexpr (WK == kWInvEuclid) return rsqrtf(d2 + kInvEps2);
    else return cauchy_w_fast(d2, inv_g2);
}

template <int WK>
__device__ __forceinline__ float2 weight_fast2(float2 d2, float2 m, float2 inv_g2) {
    if constexpr (WK == kWSoftmax) {
        const float2 t = mul2(sub2(m, d2), inv_g2);
        return make_float2(__expf(t.x), __expf(t.y));
    } else if constexpr (WK == kWInvEuclid) {
        const float2 t = add2(d2, dup2(kInvEps2));
        return make_float2(rsqrtf(t.x), rsqrtf(t.y));
    } else {
        return cauchy_w2(d2, inv_g2);
    }
}

// Factor that moves sums taken with shift m_old onto shift m_new <= m_old
// (exactly 1 when the shift did not move, 0 when nothing was summed yet).
__device__ __forceinline__ float shift_scale(float m_new, float m_old, float inv_g2) {
    return m_new == m_old ? 1.f : __expf((m_new - m_old) * inv_g2);
}

}  // namespace zeta
